// UltraQuant head_dim=256 4-bit paged decode: split-KV partition kernel and
// combine + un-rotation kernel.
//
// What it computes follows the vLLM ultraquant_decode_hd256 page (PR 59857):
//  * slot cache [num_blocks][block_size][Hk][padded_slot] uint8 with K e2m1
//    codes (bytes 0..127, dim 2i in the low nibble of byte i), K scales
//    (128..135, one per 32 dims), V codes (136..263) and V scales (264..271)
//    -- builder docstring and STEP F offsets;
//  * in-kernel Walsh-Hadamard rotation of Q, q_r = q H / 16 (STEP B'), and
//    attention in the rotated domain with softmax scale 1/sqrt(256);
//  * tile groups of 256 tokens strided over partitions (STEP F), partials
//    (O, m, l) per (seq, kv_head, partition) (STEP G);
//  * the combine merges partitions and rotates the output back (o = o_r H/16).
// Readings: the group scales are e4m3 and V decodes through a 16-entry fp32
// centroid table (V = centroid[code] * scale); the page's own V convert
// (e2m1 * scale) is the case where the table is the e2m1 value table.
//
// GB300 design: the fp8 kernel's structure (persistent 4-warp CTAs, per-warp
// 16-byte cp.async pipelines, deterministic merge) with
//  * K dequantised in registers: cvt e2m1x2 -> f16x2 (exact) times the
//    group scale (hmul2, exact in f16), f16 mma.sync against the rotated q;
//  * V^T fragments built per token pair: the two tokens' nibbles of a dim form
//    one byte that indexes a 256-entry f16x2 table {c[a], c[b]} in shared
//    memory (replicated per bank, conflict-free), times the token pair's
//    scale; when the centroid table is exactly the e2m1 table the byte is
//    converted with cvt e2m1x2 instead (detected in the kernel);
//  * a lane's 32 output dims form one scale group, so one scale pair serves
//    all of its V fragments of a token pair.
#include "common.cuh"
#include "qpa_internal.h"
#include "combine.cuh"

namespace qpa {

namespace uq {
constexpr int D = 256;
constexpr int TG = 256;
constexpr int SLICE = 16;
constexpr int NW = 4;
constexpr int THREADS = NW * 32;
constexpr int DEPTH = 4;
constexpr int CONTENT = 272;                     // used bytes of a slot
constexpr int SLOT_BYTES = SLICE * CONTENT;      // 4352: one slice, or 8 query rows (4096)
constexpr int KS_OFF = 128, VC_OFF = 136, VS_OFF = 264;
constexpr int LUT_BYTES = 256 * 32 * 4;          // [code pair][bank copy] f16x2
constexpr int ringOff = 0;
constexpr int lutOff = NW * DEPTH * SLOT_BYTES;  // 69632 (a multiple of 128)
constexpr int mOff = lutOff + LUT_BYTES;
constexpr int lOff = mOff + NW * 8 * 4;
constexpr int fOff = lOff + NW * 8 * 4;
constexpr int SMEM = fOff + NW * 4;
constexpr int CTAS_PER_SM = 2;
}  // namespace uq

struct UqParams {
  const uint16_t* q;
  const uint8_t* kv;
  const float* centroids;
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* part_o;
  float* part_m;
  float* part_l;
  long long q_stride_seq, q_stride_head;
  int num_seqs, num_kv_heads, qg, block_size, log2_bs, num_blocks, max_blocks, num_partitions, padded_slot;
  float softmax_scale;
};

enum : int { UEV_NONE = 0, UEV_ITEM = 1, UEV_SLICE = 2 };

// e2m1 values in code order (the table for which V decodes with cvt).
__device__ __forceinline__ float e2m1_value(int k) {
  const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  return (k & 8) ? -mag[k & 7] : mag[k & 7];
}

__global__ void __launch_bounds__(uq::THREADS, uq::CTAS_PER_SM)
uq_partition_kernel(const UqParams p) {
  using namespace uq;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_items = p.num_seqs * p.num_kv_heads * p.num_partitions;
  const int P = p.num_partitions;
  const int bs = p.block_size;
  const int lbs = p.log2_bs;
  const int bpt = TG / bs > 0 ? TG / bs : 1;
  float* ms = reinterpret_cast<float*>(smem + mOff);
  float* ls = reinterpret_cast<float*>(smem + lOff);
  uint32_t* fslot = reinterpret_cast<uint32_t*>(smem + fOff);
  const uint32_t lut = smem_u32(smem + lutOff) + lane * 4;   // this lane's bank copy

  // ---- centroid table: the e2m1 table takes the cvt path, anything else the
  // shared-memory pair table (f16 values of the fp32 centroids)
  bool e2m1_table = true;
  {
    float cv[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      cv[k] = __ldg(p.centroids + k);
      e2m1_table = e2m1_table && (cv[k] == e2m1_value(k)) && (__float_as_uint(cv[k]) >> 31) == (uint32_t)(k >> 3);
    }
    if (!e2m1_table) {
      uint32_t* t = reinterpret_cast<uint32_t*>(smem + lutOff);
      for (int i = threadIdx.x; i < 256 * 32; i += THREADS) {
        const int e = i >> 5;
        t[i] = f32x2_to_f16x2(cv[e & 15], cv[e >> 4]);
      }
    }
  }
  __syncthreads();
  pdl_launch_dependents();

  const uint64_t pol = policy_evict_first();
  const uint32_t ring = smem_u32(smem + ringOff) + warp * DEPTH * SLOT_BYTES;
  const size_t tok_stride = size_t(p.num_kv_heads) * p.padded_slot;    // bytes between tokens

  // ---------------------------------------------------------------- issue side
  int ik_item = blockIdx.x;
  int i_state = 0, i_tg = 0, i_kk = 0, i_L = 0, i_Lnext = 0, i_seq = 0, i_kvh = 0, i_part = 0;
  int32_t i_ent = 0, i_nent = 0;
  int rec_kind = 0, rec_a = 0, rec_b = 0;

  auto load_len = [&](int item) -> int {
    if (item >= num_items) return 0;
    const int seq = item / (P * p.num_kv_heads);
    return max(0, min(__ldg(p.seq_lens + seq), p.max_blocks * bs));
  };
  auto load_entries = [&](int seq, int tg, int L) -> int32_t {
    const int e = tg * bpt + lane;
    int32_t v = 0;
    if (lane < bpt && (e << lbs) < L) v = __ldg(p.block_table + (long long)seq * p.max_blocks + e);
    return v;
  };
  if (ik_item < num_items) i_L = load_len(ik_item);
  i_Lnext = load_len(ik_item + gridDim.x);

  auto issue = [&](int e) {
    const uint32_t slot = ring + (e % DEPTH) * SLOT_BYTES;
    int kind = UEV_NONE, a = 0, b = 0;
    while (true) {
      if (ik_item >= num_items) break;
      if (i_state == 0) {
        i_part = ik_item % P;
        const int t = ik_item / P;
        i_kvh = t % p.num_kv_heads;
        i_seq = t / p.num_kv_heads;
        if (i_part * TG < i_L) {
          // query rows: qg rows x 512 B
          const uint16_t* qrow0 = p.q + i_seq * p.q_stride_seq + (long long)(i_kvh * p.qg) * p.q_stride_head;
          for (int idx = lane; idx < p.qg * 32; idx += 32) {
            const int row = idx >> 5, ch = idx & 31;
            cp_async16(slot + row * 512 + ch * 16, qrow0 + row * p.q_stride_head + ch * 8, pol);
          }
          i_ent = load_entries(i_seq, i_part, i_L);
          if ((i_part + P) * TG < i_L) i_nent = load_entries(i_seq, i_part + P, i_L);
        }
        i_state = 1;
        i_tg = i_part;
        i_kk = 0;
        kind = UEV_ITEM; a = ik_item; b = i_L;
        break;
      }
      if (i_tg * TG >= i_L) {
        ik_item += gridDim.x;
        i_state = 0;
        i_L = i_Lnext;
        i_Lnext = load_len(ik_item + gridDim.x);
        continue;
      }
      const int s = (i_tg * TG) / SLICE + 4 * i_kk + warp;
      const bool valid = s * SLICE < i_L;
      int phys = __shfl_sync(0xffffffffu, i_ent, ((s * SLICE) & (TG - 1)) >> lbs);
      if (++i_kk == 4) {
        i_kk = 0;
        i_tg += P;
        if (i_tg * TG < i_L) {
          i_ent = i_nent;
          if ((i_tg + P) * TG < i_L) i_nent = load_entries(i_seq, i_tg + P, i_L);
        }
      }
      if (!valid) continue;
      if (phys < 0 || phys >= p.num_blocks) {
        if (lane == 0) atomicExch(&g_kernel_error, KERR_BAD_BLOCK);
        phys = 0;
      }
      // 16 token slots of this KV head, 272 bytes each: lanes 2r and 2r+1 copy
      // the alternate 16-byte chunks of token r
      const uint8_t* tok = p.kv + (size_t(phys) * bs + ((s * SLICE) & (bs - 1)) + (lane >> 1)) * tok_stride +
                           size_t(i_kvh) * p.padded_slot + 16 * (lane & 1);
      cp_async_slot272(slot + (lane >> 1) * CONTENT + 16 * (lane & 1), tok, (lane & 1) == 0, pol);
      kind = UEV_SLICE; a = s; b = i_L;
      break;
    }
    cp_async_commit();
    if (lane == e % DEPTH) { rec_kind = kind; rec_a = a; rec_b = b; }
  };

  // ---------------------------------------------------------------- consume side
  const int g = lane >> 2;
  const int c = lane & 3;
  const float rowc = p.softmax_scale * kLog2e;
  uint32_t qf[32];          // rotated query row g, dims [64c, 64c+64), f16x2
  float o[16][4];           // O^T: m-tile i rows g, g+8 = dims 32g+2i, 32g+2i+1
  float m_run[2], l_run[2];
  int cur_item = -1;

#pragma unroll 1
  for (int e = 0; e < DEPTH - 1; ++e) issue(e);

#pragma unroll 1
  for (int e = 0;; ++e) {
    const int kind = __shfl_sync(0xffffffffu, rec_kind, e % DEPTH);
    const int ea = __shfl_sync(0xffffffffu, rec_a, e % DEPTH);
    const int eb = __shfl_sync(0xffffffffu, rec_b, e % DEPTH);

    if (kind != UEV_SLICE && cur_item >= 0) {
      // ---- merge the four warps' states (fixed order), write partials
      const long long row0 = (long long)cur_item * p.qg;
      const uint32_t myfree = ring + ((e + DEPTH - 1) % DEPTH) * SLOT_BYTES;
#pragma unroll
      for (int sh = 4; sh < 32; sh <<= 1) {
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], sh);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], sh);
      }
      if (g == 0) {
        ms[warp * 8 + 2 * c] = m_run[0];
        ms[warp * 8 + 2 * c + 1] = m_run[1];
        ls[warp * 8 + 2 * c] = l_run[0];
        ls[warp * 8 + 2 * c + 1] = l_run[1];
      }
      if (lane == 0) fslot[warp] = myfree;
      named_barrier(1, THREADS);
      float sc[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, ms[w * 8 + 2 * c + h]);
        sc[h] = (m_run[h] == -INFINITY) ? 0.f : ex2(m_run[h] - M);
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        // dims [128 half, 128 half + 128) are held by lanes with g in [4 half, 4 half + 4);
        // stored as fp32 [8 rows][128] with bits 1..4 of the dim XOR-swizzled
        if ((g >> 2) == half) {
          const int gg = g & 3;
          const int sw = ((c | (gg << 2)) << 1);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int d0 = 32 * gg + 2 * i;     // local dim of row g (even), +1 for row g+8
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int row = 2 * c + h;
              stsf(myfree + (row * 128 + (d0 ^ sw)) * 4, o[i][h] * sc[h]);
              stsf(myfree + (row * 128 + ((d0 + 1) ^ sw)) * 4, o[i][2 + h] * sc[h]);
            }
          }
        }
        named_barrier(1, THREADS);
        {
          const int tid = threadIdx.x;
          uint32_t fs[NW];
#pragma unroll
          for (int w = 0; w < NW; ++w) fs[w] = fslot[w];
          for (int r = 0; r < p.qg; ++r) {
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NW; ++w) M = fmaxf(M, ms[w * 8 + r]);
            float lsum = 0.f, acc = 0.f;
            const int pd = tid ^ ((((r >> 1) | (((tid >> 5) & 3) << 2))) << 1);
#pragma unroll
            for (int w = 0; w < NW; ++w) {
              const float mw = ms[w * 8 + r];
              const float wt = (mw == -INFINITY) ? 0.f : ex2(mw - M);
              lsum += wt * ls[w * 8 + r];
              acc += ldsf(fs[w] + (r * 128 + pd) * 4);
            }
            p.part_o[(row0 + r) * D + 128 * half + tid] = lsum > 0.f ? acc / lsum : 0.f;
            if (half == 0 && tid == 0) {
              p.part_m[row0 + r] = M == -INFINITY ? -INFINITY : M * kLn2;
              p.part_l[row0 + r] = lsum;
            }
          }
        }
        named_barrier(1, THREADS);
      }
      cur_item = -1;
    }

    if (kind == UEV_NONE) break;
    issue(e + DEPTH - 1);
    cp_async_wait<DEPTH - 1>();
    __syncwarp();
    const uint32_t slot = ring + (e % DEPTH) * SLOT_BYTES;

    if (kind == UEV_ITEM) {
      cur_item = ea;
      const bool work = (ea % P) * TG < eb;
      // ---- rotated query: row g, dims [64c, 64c+64); butterfly stages with
      // strides 1..32 in registers, 64 and 128 across lanes c^1 and c^2
      float v[64];
      if (work && g < p.qg) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 w4 = lds128(slot + g * 512 + c * 128 + j * 16);
          const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            v[8 * j + 2 * k] = __uint_as_float(ws[k] << 16);
            v[8 * j + 2 * k + 1] = __uint_as_float(ws[k] & 0xffff0000u);
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < 64; ++k) v[k] = 0.f;
      }
#pragma unroll
      for (int st = 1; st < 64; st <<= 1) {
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          if ((k & st) == 0) {
            const float x = v[k], y = v[k + st];
            v[k] = x + y;
            v[k + st] = x - y;
          }
        }
      }
#pragma unroll
      for (int sh = 1; sh <= 2; sh <<= 1) {
        const bool upper = (c & sh) != 0;
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          const float pv = __shfl_xor_sync(0xffffffffu, v[k], sh);
          v[k] = upper ? pv - v[k] : v[k] + pv;
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) qf[j] = f32x2_to_f16x2(v[2 * j] * 0.0625f, v[2 * j + 1] * 0.0625f);
      m_run[0] = m_run[1] = -INFINITY;
      l_run[0] = l_run[1] = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) o[i][k] = 0.f;
      __syncwarp();
      continue;
    }

    // ---- UEV_SLICE: tokens [16 ea, 16 ea + 16)
    const int t0 = ea * SLICE;
    const int L = eb;
    const bool partial = t0 + SLICE > L;
    // K: rows g and g+8, code bytes [32c, 32c+32) -> dims [64c, 64c+64)
    const uint32_t rg = slot + g * CONTENT, rg8 = slot + (g + 8) * CONTENT;
    const uint4 ka0 = lds128(rg + 32 * c), ka1 = lds128(rg + 32 * c + 16);
    const uint4 kb0 = lds128(rg8 + 32 * c), kb1 = lds128(rg8 + 32 * c + 16);
    const uint32_t kra[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
    const uint32_t krb[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
    // K scales of groups 2c, 2c+1 for rows g, g+8 as {s, s} f16 pairs
    uint32_t ksa0, ksa1, ksb0, ksb1;
    {
      const uint32_t sa = e4m3x2_lo_to_f16x2(lds32(rg + KS_OFF + 4 * (c >> 1)) >> (16 * (c & 1)));
      const uint32_t sb = e4m3x2_lo_to_f16x2(lds32(rg8 + KS_OFF + 4 * (c >> 1)) >> (16 * (c & 1)));
      ksa0 = prmt(sa, sa, 0x1010); ksa1 = prmt(sa, sa, 0x3232);
      ksb0 = prmt(sb, sb, 0x1010); ksb1 = prmt(sb, sb, 0x3232);
    }
    // V: rows 2c, 2c+1, 2c+8, 2c+9, code bytes [16g, 16g+16) -> dims [32g, 32g+32)
    uint2 vw[4][2];
    uint32_t vsc;     // V scale bytes of group g for rows 2c, 2c+1, 2c+8, 2c+9
    {
      const int rows[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
      uint32_t sbytes[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t rb = slot + rows[j] * CONTENT;
        vw[j][0] = lds64(rb + VC_OFF + 16 * g);
        vw[j][1] = lds64(rb + VC_OFF + 16 * g + 8);
        sbytes[j] = lds32(rb + VS_OFF + 4 * (g >> 2)) >> (8 * (g & 3));
      }
      vsc = prmt(prmt(sbytes[0], sbytes[1], 0x0040), prmt(sbytes[2], sbytes[3], 0x0040), 0x5410);
    }
    if (partial) {
      // tokens past the end may hold NaN scale bytes: zero their V words and scales
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tok = t0 + 2 * c + (j & 1) + 8 * (j >> 1);
        if (tok >= L) {
          vw[j][0] = make_uint2(0, 0);
          vw[j][1] = make_uint2(0, 0);
          vsc &= ~(0xffu << (8 * j));
        }
      }
    }
    const uint32_t vs01 = e4m3x2_lo_to_f16x2(vsc);    // {s[2c], s[2c+1]}
    const uint32_t vs89 = e4m3x2_hi_to_f16x2(vsc);    // {s[2c+8], s[2c+9]}

    // ---- S^T (16 tokens x 8 rows) = K q_r^T
    float sa4[4] = {0.f, 0.f, 0.f, 0.f}, sb4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t sA = j < 4 ? ksa0 : ksa1, sB = j < 4 ? ksb0 : ksb1;
      const uint32_t a00 = hmul2(e2m1x2_to_f16x2<0>(kra[j]), sA), a01 = hmul2(e2m1x2_to_f16x2<1>(kra[j]), sA);
      const uint32_t a02 = hmul2(e2m1x2_to_f16x2<2>(kra[j]), sA), a03 = hmul2(e2m1x2_to_f16x2<3>(kra[j]), sA);
      const uint32_t b00 = hmul2(e2m1x2_to_f16x2<0>(krb[j]), sB), b01 = hmul2(e2m1x2_to_f16x2<1>(krb[j]), sB);
      const uint32_t b02 = hmul2(e2m1x2_to_f16x2<2>(krb[j]), sB), b03 = hmul2(e2m1x2_to_f16x2<3>(krb[j]), sB);
      // k-step 2j: dims 64c+8j+{0,1} | {2,3}; k-step 2j+1: dims +{4,5} | {6,7}
      mma_f16_16816(sa4, a00, b00, a01, b01, qf[4 * j], qf[4 * j + 1]);
      mma_f16_16816(sb4, a02, b02, a03, b03, qf[4 * j + 2], qf[4 * j + 3]);
    }
    float x0 = (sa4[0] + sb4[0]) * rowc, x1 = (sa4[1] + sb4[1]) * rowc;
    float x2 = (sa4[2] + sb4[2]) * rowc, x3 = (sa4[3] + sb4[3]) * rowc;
    if (partial) {
      if (t0 + g >= L) { x0 = -INFINITY; x1 = -INFINITY; }
      if (t0 + g + 8 >= L) { x2 = -INFINITY; x3 = -INFINITY; }
    }
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
    }
    const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
    if (__any_sync(0xffffffffu, (mn0 > m_run[0]) || (mn1 > m_run[1]))) {
      const float a0 = ex2(m_run[0] - mn0), a1 = ex2(m_run[1] - mn1);
      l_run[0] *= a0;
      l_run[1] *= a1;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[i][0] *= a0; o[i][1] *= a1;
        o[i][2] *= a0; o[i][3] *= a1;
      }
      m_run[0] = mn0;
      m_run[1] = mn1;
    }
    const float p0 = ex2(x0 - mn0), p1 = ex2(x1 - mn1);
    const float p2 = ex2(x2 - mn0), p3 = ex2(x3 - mn1);
    const uint32_t P01 = f32x2_to_f16x2(p0, p1);
    const uint32_t P23 = f32x2_to_f16x2(p2, p3);
    l_run[0] += f16_lo_to_f32(P01) + f16_lo_to_f32(P23);
    l_run[1] += f16_hi_to_f32(P01) + f16_hi_to_f32(P23);
    const uint32_t b0 = movmatrix_trans(P01);
    const uint32_t b1 = movmatrix_trans(P23);

    // ---- O^T += V^T P^T. For byte i of the lane's 16 V-code bytes, the low
    // nibbles of tokens (2c, 2c+1) form index E (dim 32g+2i, m-tile i row g) and
    // the high nibbles index O (dim 32g+2i+1, row g+8); likewise tokens 2c+8, 2c+9.
#pragma unroll
    for (int wq = 0; wq < 4; ++wq) {          // 4 code bytes (m-tiles 4wq..4wq+3) per word
      const uint32_t w0 = wq < 2 ? (wq == 0 ? vw[0][0].x : vw[0][0].y) : (wq == 2 ? vw[0][1].x : vw[0][1].y);
      const uint32_t w1 = wq < 2 ? (wq == 0 ? vw[1][0].x : vw[1][0].y) : (wq == 2 ? vw[1][1].x : vw[1][1].y);
      const uint32_t w8 = wq < 2 ? (wq == 0 ? vw[2][0].x : vw[2][0].y) : (wq == 2 ? vw[2][1].x : vw[2][1].y);
      const uint32_t w9 = wq < 2 ? (wq == 0 ? vw[3][0].x : vw[3][0].y) : (wq == 2 ? vw[3][1].x : vw[3][1].y);
      // index bytes: token pair (2c, 2c+1) even/odd dims, token pair (2c+8, 2c+9)
      const uint32_t Ea = (w0 & 0x0F0F0F0Fu) | ((w1 & 0x0F0F0F0Fu) << 4);
      const uint32_t Oa = ((w0 >> 4) & 0x0F0F0F0Fu) | (w1 & 0xF0F0F0F0u);
      const uint32_t Eb = (w8 & 0x0F0F0F0Fu) | ((w9 & 0x0F0F0F0Fu) << 4);
      const uint32_t Ob = ((w8 >> 4) & 0x0F0F0F0Fu) | (w9 & 0xF0F0F0F0u);
      uint32_t fa[4][4];    // [byte][a0 a1 a2 a3]
      if (e2m1_table) {
        fa[0][0] = e2m1x2_to_f16x2<0>(Ea); fa[0][1] = e2m1x2_to_f16x2<0>(Oa);
        fa[0][2] = e2m1x2_to_f16x2<0>(Eb); fa[0][3] = e2m1x2_to_f16x2<0>(Ob);
        fa[1][0] = e2m1x2_to_f16x2<1>(Ea); fa[1][1] = e2m1x2_to_f16x2<1>(Oa);
        fa[1][2] = e2m1x2_to_f16x2<1>(Eb); fa[1][3] = e2m1x2_to_f16x2<1>(Ob);
        fa[2][0] = e2m1x2_to_f16x2<2>(Ea); fa[2][1] = e2m1x2_to_f16x2<2>(Oa);
        fa[2][2] = e2m1x2_to_f16x2<2>(Eb); fa[2][3] = e2m1x2_to_f16x2<2>(Ob);
        fa[3][0] = e2m1x2_to_f16x2<3>(Ea); fa[3][1] = e2m1x2_to_f16x2<3>(Oa);
        fa[3][2] = e2m1x2_to_f16x2<3>(Eb); fa[3][3] = e2m1x2_to_f16x2<3>(Ob);
      } else {
#pragma unroll
        for (int bq = 0; bq < 4; ++bq) {
          fa[bq][0] = lds32(lut + (((Ea >> (8 * bq)) & 0xFFu) << 7));
          fa[bq][1] = lds32(lut + (((Oa >> (8 * bq)) & 0xFFu) << 7));
          fa[bq][2] = lds32(lut + (((Eb >> (8 * bq)) & 0xFFu) << 7));
          fa[bq][3] = lds32(lut + (((Ob >> (8 * bq)) & 0xFFu) << 7));
        }
      }
#pragma unroll
      for (int bq = 0; bq < 4; ++bq) {
        const int i = 4 * wq + bq;
        mma_f16_16816(o[i], hmul2(fa[bq][0], vs01), hmul2(fa[bq][1], vs01), hmul2(fa[bq][2], vs89),
                      hmul2(fa[bq][3], vs89), b0, b1);
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
}

// Combine the partitions of one query row (combine_row) and rotate it back:
// out = o_r H/16, 8 butterfly stages over the 256 dims, one pair per thread.
template <typename OutT>
__global__ void __launch_bounds__(kCombineThreads)
uq_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_m,
                  const float* __restrict__ part_l, OutT* __restrict__ out, int num_kv_heads, int qg,
                  int num_partitions, long long out_stride_seq, long long out_stride_head) {
  constexpr int D = 256;
  extern __shared__ __align__(16) float sw[];
  __shared__ __align__(16) float vec[D];
  pdl_wait_primary();
  const int row = blockIdx.x;
  const int r = row % qg;
  const int sk = row / qg;
  const int seq = sk / num_kv_heads, kvh = sk % num_kv_heads;
  const int tid = threadIdx.x;
  combine_row<D>(part_o, part_m, part_l, (long long)sk * num_partitions * qg + r, qg, num_partitions, sw, vec);
  for (int st = 1; st < D; st <<= 1) {
    const int i = ((tid & ~(st - 1)) << 1) | (tid & (st - 1));   // index with bit `st` clear
    const float x = vec[i], y = vec[i + st];
    __syncthreads();
    vec[i] = x + y;
    vec[i + st] = x - y;
    __syncthreads();
  }
  if (tid < D / 4) {
    OutT* dst = out + seq * out_stride_seq + (long long)(kvh * qg + r) * out_stride_head + 4 * tid;
    store4(dst, vec[4 * tid] * 0.0625f, vec[4 * tid + 1] * 0.0625f, vec[4 * tid + 2] * 0.0625f,
           vec[4 * tid + 3] * 0.0625f);
  }
}

// ------------------------------------------------------------------ host side
cudaError_t launch_uq_partition(const UqLaunch& a, cudaStream_t stream) {
  UqParams p;
  p.q = static_cast<const uint16_t*>(a.q);
  p.kv = a.kv;
  p.centroids = a.centroids;
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  p.part_o = a.part_o;
  p.part_m = a.part_m;
  p.part_l = a.part_l;
  p.q_stride_seq = a.q_stride_seq;
  p.q_stride_head = a.q_stride_head;
  p.num_seqs = a.num_seqs;
  p.num_kv_heads = a.num_kv_heads;
  p.qg = a.qg;
  p.block_size = a.block_size;
  p.log2_bs = 0;
  while ((1 << p.log2_bs) < a.block_size) ++p.log2_bs;
  p.num_blocks = a.num_blocks;
  p.max_blocks = a.max_blocks;
  p.num_partitions = a.num_partitions;
  p.padded_slot = a.padded_slot;
  p.softmax_scale = a.softmax_scale;
  const long long items = (long long)a.num_seqs * a.num_kv_heads * a.num_partitions;
  if (items <= 0) return cudaSuccess;
  const int grid = (int)std::min<long long>(items, (long long)uq::CTAS_PER_SM * a.num_sms);
  cudaFuncSetAttribute(uq_partition_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, uq::SMEM);
  uq_partition_kernel<<<grid, uq::THREADS, uq::SMEM, stream>>>(p);
  return cudaGetLastError();
}

template <typename OutT>
static cudaError_t launch_uq_combine_t(const CombineLaunch& a, OutT* out, cudaStream_t stream) {
  const int grid = a.num_seqs * a.num_kv_heads * a.qg;
  const size_t smem = combine_smem_bytes(a.num_partitions);
  if (smem > 40 * 1024)
    cudaFuncSetAttribute(uq_combine_kernel<OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, uq_combine_kernel<OutT>, a.part_o, a.part_m, a.part_l, out, a.num_kv_heads,
                            a.qg, a.num_partitions, a.out_stride_seq, a.out_stride_head);
}

cudaError_t launch_uq_combine(const CombineLaunch& a, cudaStream_t stream) {
  if (a.num_seqs * a.num_kv_heads * a.qg <= 0) return cudaSuccess;
  cudaError_t e = a.out_bf16 ? launch_uq_combine_t(a, static_cast<__nv_bfloat16*>(a.out), stream)
                             : launch_uq_combine_t(a, static_cast<float*>(a.out), stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qpa
