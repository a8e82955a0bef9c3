// Flash-combine of split-KV partials for one query row ([PA] "parallel
// flash-combine reduce kernel"): M = max_p m_p, w_p = l_p exp(m_p - M),
// o = sum_p w_p O_p / sum_p w_p. An empty partition (m_p = -inf) has weight
// exactly 0; the exponent argument is clamped so no NaN can arise.
//
// One 128-thread CTA per row. The first chunk of O loads and all (m, l)
// loads are issued before any dependent work, so a row costs one global
// round trip plus one more per further chunk of 8 partitions per thread.
#pragma once
#include "common.cuh"

namespace qpa {

constexpr int kCombineThreads = 128;

// Returns in vec[0..D) (shared memory) the combined row. `sw` is dynamic
// shared scratch of at least 2*P + 4*128 floats (16-byte aligned).
template <int D>
__device__ __forceinline__ void combine_row(const float* __restrict__ part_o, const float* __restrict__ part_m,
                                            const float* __restrict__ part_l, long long rbase, int qg,
                                            int num_partitions, float* sw, float* vec) {
  constexpr int NVEC = D / 4;                  // float4 per row
  constexpr int NSUB = kCombineThreads / NVEC; // partition subsets
  constexpr int CH = 8;                        // partitions per thread per chunk
  const int P = num_partitions;
  const int tid = threadIdx.x, lane = tid & 31;
  const int v4 = tid % NVEC, sub = tid / NVEC;
  float* ms = sw;
  float* ls = sw + P;
  float4* part = reinterpret_cast<float4*>(sw + ((2 * P + 3) & ~3));
  // rbase = ((seq * Hk + kvh) * P) * qg + r: partition pp of the row is at rbase + pp * qg
  const float* ob = part_o + rbase * D + 4 * v4;
  float4 o[CH];
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    const int pp = sub + k * NSUB;
    o[k] = pp < P ? __ldg(reinterpret_cast<const float4*>(ob + (long long)pp * qg * D)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int pp = tid; pp < P; pp += kCombineThreads) {
    ms[pp] = part_m[rbase + (long long)pp * qg];
    ls[pp] = part_l[rbase + (long long)pp * qg];
  }
  __syncthreads();
  float M = -INFINITY;
  for (int pp = lane; pp < P; pp += 32) M = fmaxf(M, ms[pp]);
#pragma unroll
  for (int sh = 16; sh; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, sh));
  auto weight = [&](int pp) -> float {
    const float m = ms[pp];
    return (M == -INFINITY || m == -INFINITY) ? 0.f : ls[pp] * __expf(fmaxf(m - M, -80.f));
  };
  float den = 0.f;
  for (int pp = lane; pp < P; pp += 32) den += weight(pp);
#pragma unroll
  for (int sh = 16; sh; sh >>= 1) den += __shfl_xor_sync(0xffffffffu, den, sh);
  const float inv = den > 0.f ? 1.f / den : 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    const int pp = sub + k * NSUB;
    if (pp < P) {
      const float w = weight(pp);
      acc.x += w * o[k].x; acc.y += w * o[k].y; acc.z += w * o[k].z; acc.w += w * o[k].w;
    }
  }
  for (int base = CH * NSUB; base < P; base += CH * NSUB) {
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const int pp = base + sub + k * NSUB;
      o[k] = pp < P ? __ldg(reinterpret_cast<const float4*>(ob + (long long)pp * qg * D)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const int pp = base + sub + k * NSUB;
      if (pp < P) {
        const float w = weight(pp);
        acc.x += w * o[k].x; acc.y += w * o[k].y; acc.z += w * o[k].z; acc.w += w * o[k].w;
      }
    }
  }
  part[tid] = acc;
  __syncthreads();
  if (sub == 0) {
#pragma unroll
    for (int s = 1; s < NSUB; ++s) {
      const float4 b = part[s * NVEC + v4];
      acc.x += b.x; acc.y += b.y; acc.z += b.z; acc.w += b.w;
    }
    vec[4 * v4 + 0] = acc.x * inv;
    vec[4 * v4 + 1] = acc.y * inv;
    vec[4 * v4 + 2] = acc.z * inv;
    vec[4 * v4 + 3] = acc.w * inv;
  }
  __syncthreads();
}

inline size_t combine_smem_bytes(int num_partitions) {
  return (size_t((2 * num_partitions + 3) & ~3) + 4 * kCombineThreads) * sizeof(float);
}

}  // namespace qpa
