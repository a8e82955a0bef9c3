// Flash-combine of split-KV partials for one query row (the [PA] page's
// cross-partition reduce): M = max_p m_p, w_p = l_p exp(m_p - M),
// o = sum_p (w_p / sum_q w_q) O_p (the weights are normalised before the sum,
// so no partial sum exceeds the largest |O_p|). An empty partition (m_p = -inf or l_p = 0)
// has weight exactly 0 and its O is never read, so it need not be written;
// the exponent argument is clamped so no NaN can arise.
//
// One CTA per row: all (m, l) loads first, then the O loads of the
// partitions with a nonzero weight, all issued before any dependent work.
#pragma once
#include "common.cuh"

namespace qpa {

// Threads of a row CTA are NVEC = D/4 float4 columns times nsub partition
// subsets; thread (sub, column) takes partitions sub, sub + nsub, ... and
// issues up to KMAX of those loads at once, so that a row costs one global
// round trip when P <= nsub * KMAX. nsub grows with P up to
// kCombineMaxThreads threads.
constexpr int kCombineMaxThreads = 512;
constexpr int kCombineKmax128 = 16;     // partitions per thread and round trip, D = 128
constexpr int kCombineKmax256 = 20;     // D = 256

inline int combine_threads(int d, int kmax, int num_partitions) {
  const int nvec = d / 4;
  int nsub = (num_partitions + kmax - 1) / kmax;
  if (nsub < 1) nsub = 1;
  if (nsub > kCombineMaxThreads / nvec) nsub = kCombineMaxThreads / nvec;
  while ((nvec * nsub) % 32) ++nsub;   // whole warps: the reductions shuffle over 32 lanes
  return nvec * nsub;
}

// Returns in vec[0..D) (shared memory) the combined row. `sw` is shared
// scratch of combine_smem_bytes(P, nthr) bytes (16-byte aligned). The row is
// combined by the nthr threads tid = 0 .. nthr - 1 of a group (a whole warp
// or more); every group of the CTA calls this together (it holds CTA-wide
// barriers), each with its own row, scratch and vec.
// EAGER: the first round of O loads is issued together with the (m, l) loads
// instead of after the weights are known (one round trip instead of two, for
// rows whose slots are all written); an O of weight 0 is never used.
template <int D, int KMAX, bool EAGER = false>
__device__ __forceinline__ void combine_row(const float* __restrict__ part_o, const float* __restrict__ part_m,
                                            const float* __restrict__ part_l, long long rbase, int qg,
                                            int num_partitions, float* sw, float* vec, int tid, int nthr) {
  constexpr int NVEC = D / 4;                  // float4 per row
  const int nsub = nthr / NVEC;                // partition subsets
  const int P = num_partitions;
  const int lane = tid & 31;
  const int v4 = tid % NVEC, sub = tid / NVEC;
  float* ms = sw;
  float* ls = sw + P;
  float4* part = reinterpret_cast<float4*>(sw + ((2 * P + 3) & ~3));
  // rbase = ((seq * Hk + kvh) * P) * qg + r: partition pp of the row is at rbase + pp * qg
  const float* ob = part_o + rbase * D + 4 * v4;
  const long long pstride = (long long)qg * D;
  float4 o0[EAGER ? KMAX : 1];
  if constexpr (EAGER) {
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      const int pp = sub + k * nsub;
      o0[k] = pp < P ? __ldg(reinterpret_cast<const float4*>(ob + pp * pstride)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  for (int pp = tid; pp < P; pp += nthr) {
    ms[pp] = part_m[rbase + (long long)pp * qg];
    ls[pp] = part_l[rbase + (long long)pp * qg];
  }
  __syncthreads();
  // every warp reduces the maximum and the denominator over all partitions
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
  int base0 = 0;
  if constexpr (EAGER) {
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      const int pp = sub + k * nsub;
      const float w = pp < P ? weight(pp) * inv : 0.f;
      if (w != 0.f) {
        acc.x += w * o0[k].x; acc.y += w * o0[k].y; acc.z += w * o0[k].z; acc.w += w * o0[k].w;
      }
    }
    base0 = KMAX * nsub;
  }
  for (int base = base0; base < P; base += KMAX * nsub) {
    float w[KMAX];
    float4 o[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      const int pp = base + sub + k * nsub;
      w[k] = pp < P ? weight(pp) * inv : 0.f;     // normalised first: no partial sum exceeds max |O_p|
      o[k] = w[k] != 0.f ? __ldg(reinterpret_cast<const float4*>(ob + pp * pstride)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      acc.x += w[k] * o[k].x; acc.y += w[k] * o[k].y; acc.z += w[k] * o[k].z; acc.w += w[k] * o[k].w;
    }
  }
  part[tid] = acc;
  __syncthreads();
  if (sub == 0) {
    for (int s = 1; s < nsub; ++s) {
      const float4 b = part[s * NVEC + v4];
      acc.x += b.x; acc.y += b.y; acc.z += b.z; acc.w += b.w;
    }
    vec[4 * v4 + 0] = acc.x;
    vec[4 * v4 + 1] = acc.y;
    vec[4 * v4 + 2] = acc.z;
    vec[4 * v4 + 3] = acc.w;
  }
  __syncthreads();
}

__host__ __device__ inline size_t combine_smem_bytes(int num_partitions, int threads) {
  return (size_t((2 * num_partitions + 3) & ~3) + 4 * size_t(threads)) * sizeof(float);
}

// Rows per CTA of a multi-row combine: the largest divisor of the rows of a
// (sequence, KV head) whose thread groups fit kCombineMaxThreads, so that a
// CTA never holds a partial group.
inline int combine_rows_per_cta(int rows, int threads) {
  int best = 1;
  for (int k = 1; k <= rows; ++k)
    if (rows % k == 0 && k * threads <= kCombineMaxThreads) best = k;
  return best;
}

}  // namespace qpa
