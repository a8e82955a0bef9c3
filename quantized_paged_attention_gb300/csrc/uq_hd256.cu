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
// (e2m1 * scale) is the case where the table is the e2m1 value table. Two
// descriptor flags select the page's own formats: UE8M0 group scales
// (2^(byte-127), built as f16 from the byte placed in a float32 exponent
// field), the e4m3 rounding of softmax_scale * q_r after the rotation
// (the logits then take no further scale), and the rotation's column
// permutation (a permuted q load here, a permuted store in the combine).
//
// GB300 design: one persistent 8-warp CTA per SM; each warp runs its own
// ring of three 32-token slices (8.5 KB each) filled by tensor-map copies. An item
// (sequence, KV head, partition) belongs to a group of W warps (W = 1, 2 or
// 4, picked on the host from the item count), which split its slices and
// merge deterministically when W > 1; with W = 1 a warp writes its own
// partials and no CTA-level synchronisation remains. A slice is two 16-token
// MMA tiles, so the per-slice costs (copy issue, row-max shuffles, pipeline
// bookkeeping) are paid once per 32 tokens and the two tiles' QK chains
// overlap. And
//  * K dequantised in registers: cvt e2m1x2 -> f16x2 (exact) times the
//    group scale (hmul2, exact in f16), f16 mma.sync against the rotated q;
//  * V^T fragments built per token pair: the two tokens' nibbles of a dim form
//    one byte that indexes a 256-entry f16x2 table {c[a], c[b]} in shared
//    memory (16 bank copies: at most two lanes share a bank), times the token pair's
//    scale; when the centroid table is exactly the e2m1 table the byte is
//    converted with cvt e2m1x2 instead (detected in the kernel);
//  * a lane's 32 output dims form one scale group, so one scale pair serves
//    all of its V fragments of a token pair.
#include "qpa.h"
#include "common.cuh"
#include "qpa_internal.h"
#include "combine.cuh"
#include "tc.cuh"

namespace qpa {

namespace uq {
constexpr int D = 256;
constexpr int TG = 256;
constexpr int SLICE = 32;                        // tokens per ring slot: two 16-token MMA tiles
constexpr int NW = 8;
constexpr int THREADS = NW * 32;
constexpr int DEPTH = 3;
constexpr int CONTENT = 272;                     // used bytes of a slot
constexpr int SLOT_BYTES = SLICE * CONTENT;      // 8704: one slice, or 8 query rows (4096)
constexpr int KS_OFF = 128, VC_OFF = 136, VS_OFF = 264;
constexpr int LUT_COPIES = 16;                   // bank copies of each table entry
constexpr int LUT_BYTES = 256 * LUT_COPIES * 4;  // [code pair][bank copy] f16x2
constexpr int ringOff = 0;
constexpr int lutOff = NW * DEPTH * SLOT_BYTES;  // 208896 (a multiple of 128)
constexpr int mOff = lutOff + LUT_BYTES;
constexpr int lOff = mOff + NW * 8 * 4;
constexpr int fOff = lOff + NW * 8 * 4;
constexpr int barOff = fOff + NW * 4;            // [NW][DEPTH] slot barriers (8-byte aligned)
constexpr int abortOff = barOff + NW * DEPTH * 8;
constexpr int SMEM = abortOff + 16 + 128;        // + alignment slack: one CTA per SM
constexpr int CTAS_PER_SM = 1;
static_assert(SMEM <= 232448, "shared memory");
static_assert(barOff % 8 == 0 && SLOT_BYTES % 128 == 0, "alignment");
constexpr int TMA_ROWS = 16;                     // token rows per tensor-map box
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
  int flags;        // QPA_UQ_UE8M0_SCALES | QPA_UQ_Q_HAIRCUT
};

enum : int { UEV_NONE = 0, UEV_ITEM = 1, UEV_SLICE = 2 };

// The rotation's column permutation: the value at butterfly position d lands
// on dim rot_perm_dest(d) (bits 4, 5, 6 of the index move to 5, 6, 4);
// rot_perm_source is its inverse.
__device__ __forceinline__ int rot_perm_dest(int d) {
  return (d & 0x8F) | ((d >> 2) & 0x10) | ((d << 1) & 0x60);
}
__device__ __forceinline__ int rot_perm_source(int j) {
  return (j & 0x8F) | ((j & 0x10) << 2) | ((j >> 1) & 0x30);
}

// e2m1 values in code order (the table for which V decodes with cvt).
__device__ __forceinline__ float e2m1_value(int k) {
  const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  return (k & 8) ? -mag[k & 7] : mag[k & 7];
}

template <int W>
__global__ void __launch_bounds__(uq::THREADS, uq::CTAS_PER_SM)
uq_partition_kernel(const __grid_constant__ CUtensorMap kv_map, const UqParams p) {
  using namespace uq;
  static_assert(W == 1 || W == 2 || W == 4, "warps per item");
  constexpr int GROUPS = NW / W;              // item groups per CTA
  constexpr int SLICES_PER_WARP = TG / SLICE / W;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the tensor-map copies need 128-byte aligned destinations
  uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int grp = warp / W;                   // this warp's item group
  const int wi = warp % W;                    // rank within the group
  const int num_items = p.num_seqs * p.num_kv_heads * p.num_partitions;
  const int item_stride = gridDim.x * GROUPS;
  const int P = p.num_partitions;
  const int bs = p.block_size;
  const int lbs = p.log2_bs;
  const int bpt = TG / bs > 0 ? TG / bs : 1;
  float* ms = reinterpret_cast<float*>(smem + mOff);
  float* ls = reinterpret_cast<float*>(smem + lOff);
  uint32_t* fslot = reinterpret_cast<uint32_t*>(smem + fOff);
  uint64_t* sbar = reinterpret_cast<uint64_t*>(smem + barOff) + warp * DEPTH;   // this warp's slot barriers
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + abortOff);
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < DEPTH; ++i) mbar_init(&sbar[i], 1);
    if (warp == 0) *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 0) prefetch_tmap(&kv_map);
  const uint32_t lut = smem_u32(smem + lutOff) + (lane & (LUT_COPIES - 1)) * 4;   // this lane's bank copy

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
      for (int i = threadIdx.x; i < 256 * LUT_COPIES; i += THREADS) {
        const int e = i / LUT_COPIES;
        t[i] = f32x2_to_f16x2(cv[e & 15], cv[e >> 4]);
      }
    }
  }
  __syncthreads();
  pdl_launch_dependents();

  const uint64_t pol = policy_evict_first();
  const uint32_t ring = smem_u32(smem + ringOff) + warp * DEPTH * SLOT_BYTES;

  // ---------------------------------------------------------------- issue side
  int ik_item = blockIdx.x * GROUPS + grp;
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
  i_Lnext = load_len(ik_item + item_stride);

  // Event e of this warp's ring: lane 0 arms slot e % DEPTH's barrier with
  // the bytes it copies (query rows, or the slice's two 16-token boxes of
  // 272-byte slots through the tensor map) and issues the copies; an event
  // without copies is a plain arrival. The warp read the slot's previous
  // contents before (program order and the __syncwarp/named barriers), and
  // lane 0 orders those generic accesses before the asynchronous writes.
  auto issue = [&](int e) {
    const uint32_t slot = ring + (e % DEPTH) * SLOT_BYTES;
    uint64_t* bar = &sbar[e % DEPTH];
    int kind = UEV_NONE, a = 0, b = 0;
    bool armed = false;        // (warp-uniform) lane 0 armed the barrier with copies
    __syncwarp();
    if (lane == 0) fence_proxy_async();
    while (true) {
      if (ik_item >= num_items) break;
      if (i_state == 0) {
        // items run in (sequence, partition, KV head) order, so the groups
        // working at the same time read both heads' halves of the same token
        // records; partials are indexed (sequence, KV head, partition)
        i_kvh = ik_item % p.num_kv_heads;
        const int t = ik_item / p.num_kv_heads;
        i_part = t % P;
        i_seq = t / P;
        if (i_part * TG < i_L) {
          // query rows: qg rows x 512 B
          const uint16_t* qrow0 = p.q + i_seq * p.q_stride_seq + (long long)(i_kvh * p.qg) * p.q_stride_head;
          if (lane == 0) {
            mbar_arrive_expect_tx(bar, p.qg * 512);
            for (int row = 0; row < p.qg; ++row)
              bulk_load(slot + row * 512, qrow0 + row * p.q_stride_head, 512, bar);
          }
          armed = true;
          i_ent = load_entries(i_seq, i_part, i_L);
          if ((i_part + P) * TG < i_L) i_nent = load_entries(i_seq, i_part + P, i_L);
        }
        i_state = 1;
        i_tg = i_part;
        i_kk = 0;
        kind = UEV_ITEM; a = (i_seq * p.num_kv_heads + i_kvh) * P + i_part; b = i_L;
        break;
      }
      if (i_tg * TG >= i_L) {
        ik_item += item_stride;
        i_state = 0;
        i_L = i_Lnext;
        i_Lnext = load_len(ik_item + item_stride);
        continue;
      }
      const int s = (i_tg * TG) / SLICE + W * i_kk + wi;
      const int t0 = s * SLICE;
      const bool valid = t0 < i_L;
      // blocks of the slice's tokens 0 and 16
      int pa = __shfl_sync(0xffffffffu, i_ent, (t0 & (TG - 1)) >> lbs);
      int pb = __shfl_sync(0xffffffffu, i_ent, ((t0 + 16) & (TG - 1)) >> lbs);
      if (++i_kk == SLICES_PER_WARP) {
        i_kk = 0;
        i_tg += P;
        if (i_tg * TG < i_L) {
          i_ent = i_nent;
          if ((i_tg + P) * TG < i_L) i_nent = load_entries(i_seq, i_tg + P, i_L);
        }
      }
      if (!valid) continue;
      if (pa < 0 || pa >= p.num_blocks || pb < 0 || pb >= p.num_blocks) {
        atomicExch(&g_kernel_error, KERR_BAD_BLOCK);
        pa = (pa < 0 || pa >= p.num_blocks) ? 0 : pa;
        pb = (pb < 0 || pb >= p.num_blocks) ? 0 : pb;
      }
      // 32 token slots of this KV head, 272 bytes each: two boxes of 16 token
      // rows through the tensor map (x = the slot's 2-byte units from 0,
      // y = KV head, z = token row of the cache). Tokens 0..15 of the slice
      // lie in block pa, 16..31 in block pb (the same block unless block_size
      // is 16); slots past the end of the sequence are read from the blocks
      // the table names (or block 0) and masked by the consumer.
      if (lane == 0) {
        mbar_arrive_expect_tx(bar, SLOT_BYTES);
        tma_load_3d(slot, &kv_map, 0, i_kvh, pa * bs + (t0 & (bs - 1)), bar, pol);
        tma_load_3d(slot + TMA_ROWS * CONTENT, &kv_map, 0, i_kvh, pb * bs + ((t0 + 16) & (bs - 1)), bar, pol);
      }
      armed = true;
      kind = UEV_SLICE; a = s; b = i_L;
      break;
    }
    if (!armed && lane == 0) mbar_arrive(bar);   // no copies: the event's phase completes at once
    if (lane == e % DEPTH) { rec_kind = kind; rec_a = a; rec_b = b; }
  };

  // ---------------------------------------------------------------- consume side
  const int g = lane >> 2;
  const int c = lane & 3;
  const bool ue8m0 = (p.flags & QPA_UQ_UE8M0_SCALES) != 0;
  const bool haircut = (p.flags & QPA_UQ_Q_HAIRCUT) != 0;
  const bool rot_perm = (p.flags & QPA_UQ_ROT_PERM) != 0;
  // with the haircut the softmax scale is already inside the e4m3 query
  const float rowc = haircut ? kLog2e : p.softmax_scale * kLog2e;
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
      const long long row0 = (long long)cur_item * p.qg;
#pragma unroll
      for (int sh = 4; sh < 32; sh <<= 1) {
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], sh);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], sh);
      }
      if constexpr (W == 1) {
        // ---- the warp's own state is the item's: normalise and write
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = 2 * c + h;
          if (r < p.qg) {
            const float inv = l_run[h] > 0.f ? 1.f / l_run[h] : 0.f;
            float* dst = p.part_o + (row0 + r) * D + 32 * g;
#pragma unroll
            for (int i = 0; i < 16; ++i)
              *reinterpret_cast<float2*>(dst + 2 * i) = make_float2(o[i][h] * inv, o[i][2 + h] * inv);
            if (g == 0) {
              p.part_m[row0 + r] = m_run[h] == -INFINITY ? -INFINITY : m_run[h] * kLn2;
              p.part_l[row0 + r] = l_run[h];
            }
          }
        }
      } else {
        // ---- merge the group's W warp states (fixed order) through their
        // just-consumed ring slots, write partials
        const uint32_t myfree = ring + ((e + DEPTH - 1) % DEPTH) * SLOT_BYTES;
        const int w0 = grp * W;
        const int bar = 1 + grp;
        if (g == 0) {
          ms[warp * 8 + 2 * c] = m_run[0];
          ms[warp * 8 + 2 * c + 1] = m_run[1];
          ls[warp * 8 + 2 * c] = l_run[0];
          ls[warp * 8 + 2 * c + 1] = l_run[1];
        }
        if (lane == 0) fslot[warp] = myfree;
        named_barrier(bar, 32 * W);
        float sc[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < W; ++w) M = fmaxf(M, ms[(w0 + w) * 8 + 2 * c + h]);
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
          named_barrier(bar, 32 * W);
          {
            uint32_t fs[W];
#pragma unroll
            for (int w = 0; w < W; ++w) fs[w] = fslot[w0 + w];
            for (int r = 0; r < p.qg; ++r) {
              float M = -INFINITY;
#pragma unroll
              for (int w = 0; w < W; ++w) M = fmaxf(M, ms[(w0 + w) * 8 + r]);
              float lsum = 0.f;
#pragma unroll
              for (int w = 0; w < W; ++w) {
                const float mw = ms[(w0 + w) * 8 + r];
                lsum += ((mw == -INFINITY) ? 0.f : ex2(mw - M)) * ls[(w0 + w) * 8 + r];
              }
#pragma unroll
              for (int d = wi * 32 + lane; d < 128; d += 32 * W) {
                const int pd = d ^ ((((r >> 1) | ((d >> 5) << 2))) << 1);
                float acc = 0.f;
#pragma unroll
                for (int w = 0; w < W; ++w) acc += ldsf(fs[w] + (r * 128 + pd) * 4);
                p.part_o[(row0 + r) * D + 128 * half + d] = lsum > 0.f ? acc / lsum : 0.f;
              }
              if (half == 0 && wi == 0 && lane == 0) {
                p.part_m[row0 + r] = M == -INFINITY ? -INFINITY : M * kLn2;
                p.part_l[row0 + r] = lsum;
              }
            }
          }
          named_barrier(bar, 32 * W);
        }
      }
      cur_item = -1;
    }

    if (kind == UEV_NONE) break;
    issue(e + DEPTH - 1);
    if (!warp_wait(&sbar[e % DEPTH], (e / DEPTH) & 1, abort_flag, KERR_TIMEOUT_FULL)) {
      // give the copies still in flight a bounded time to land before the
      // CTA's shared memory goes away
      for (int d = 0; d < DEPTH; ++d) mbar_wait(&sbar[(e + d) % DEPTH], ((e + d) / DEPTH) & 1, KERR_TIMEOUT_FULL);
      break;
    }
    const uint32_t slot = ring + (e % DEPTH) * SLOT_BYTES;

    if (kind == UEV_ITEM) {
      cur_item = ea;
      const bool work = (ea % P) * TG < eb;
      // ---- rotated query: row g, dims [64c, 64c+64); butterfly stages with
      // strides 1..32 in registers, 64 and 128 across lanes c^1 and c^2. With
      // the column-permuted rotation, position m takes q[perm^-1(m)] (the
      // permutation moves index bits 4..6 only, so it commutes through the
      // Hadamard and 8-dim runs stay contiguous).
      float v[64];
      if (work && g < p.qg) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int m = 64 * c + 8 * j;
          const int src = rot_perm ? rot_perm_source(m) : m;
          const uint4 w4 = lds128(slot + g * 512 + src * 2);
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
      if (haircut) {
        // e4m3(softmax_scale * q_r), nearest even, saturating; e4m3 -> f16 is exact
#pragma unroll
        for (int j = 0; j < 32; ++j)
          qf[j] = e4m3x2_lo_to_f16x2(f32x2_to_e4m3x2(v[2 * j] * 0.0625f * p.softmax_scale,
                                                     v[2 * j + 1] * 0.0625f * p.softmax_scale));
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) qf[j] = f32x2_to_f16x2(v[2 * j] * 0.0625f, v[2 * j + 1] * 0.0625f);
      }
      m_run[0] = m_run[1] = -INFINITY;
      l_run[0] = l_run[1] = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) o[i][k] = 0.f;
      __syncwarp();
      continue;
    }

    // ---- UEV_SLICE: tokens [32 ea, 32 ea + 32) as two 16-token tiles h
    const int t0 = ea * SLICE;
    const int L = eb;
    const bool partial = t0 + SLICE > L;

    // ---- S^T (16 tokens x 8 rows) = K q_r^T per tile; the two tiles' MMA
    // chains are independent
    float x[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      // K: rows g and g+8 of tile h, code bytes [32c, 32c+32) -> dims [64c, 64c+64)
      const uint32_t rg = slot + (16 * h + g) * CONTENT, rg8 = rg + 8 * CONTENT;
      const uint4 ka0 = lds128(rg + 32 * c), ka1 = lds128(rg + 32 * c + 16);
      const uint4 kb0 = lds128(rg8 + 32 * c), kb1 = lds128(rg8 + 32 * c + 16);
      const uint32_t kra[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
      const uint32_t krb[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
      // K scales of groups 2c, 2c+1 for rows g, g+8 as {s, s} f16 pairs
      const uint32_t swa = lds32(rg + KS_OFF + 4 * (c >> 1)) >> (16 * (c & 1));
      const uint32_t swb = lds32(rg8 + KS_OFF + 4 * (c >> 1)) >> (16 * (c & 1));
      const uint32_t sa = ue8m0 ? ue8m0x2_lo_to_f16x2(swa) : e4m3x2_lo_to_f16x2(swa);
      const uint32_t sb = ue8m0 ? ue8m0x2_lo_to_f16x2(swb) : e4m3x2_lo_to_f16x2(swb);
      const uint32_t ksa0 = prmt(sa, sa, 0x1010), ksa1 = prmt(sa, sa, 0x3232);
      const uint32_t ksb0 = prmt(sb, sb, 0x1010), ksb1 = prmt(sb, sb, 0x3232);
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
#pragma unroll
      for (int r = 0; r < 4; ++r) x[h][r] = (sa4[r] + sb4[r]) * rowc;
      if (partial) {
        if (t0 + 16 * h + g >= L) { x[h][0] = -INFINITY; x[h][1] = -INFINITY; }
        if (t0 + 16 * h + g + 8 >= L) { x[h][2] = -INFINITY; x[h][3] = -INFINITY; }
      }
    }

    // ---- online softmax over the 32 tokens (rows 2c, 2c+1 of this lane)
    float mx0 = fmaxf(fmaxf(x[0][0], x[0][2]), fmaxf(x[1][0], x[1][2]));
    float mx1 = fmaxf(fmaxf(x[0][1], x[0][3]), fmaxf(x[1][1], x[1][3]));
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
    uint32_t bP[2][2];      // P^T B fragments per tile (tokens 2c.., 2c+8.. x row g)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t P01 = f32x2_to_f16x2(ex2(x[h][0] - mn0), ex2(x[h][1] - mn1));
      const uint32_t P23 = f32x2_to_f16x2(ex2(x[h][2] - mn0), ex2(x[h][3] - mn1));
      l_run[0] += f16_lo_to_f32(P01) + f16_lo_to_f32(P23);
      l_run[1] += f16_hi_to_f32(P01) + f16_hi_to_f32(P23);
      bP[h][0] = movmatrix_trans(P01);
      bP[h][1] = movmatrix_trans(P23);
    }

    // ---- O^T += V^T P^T per tile. For byte i of the lane's 16 V-code bytes,
    // the low nibbles of tokens (2c, 2c+1) form index E (dim 32g+2i, m-tile i
    // row g) and the high nibbles index O (dim 32g+2i+1, row g+8); likewise
    // tokens 2c+8, 2c+9.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      // V: rows 2c, 2c+1, 2c+8, 2c+9 of tile h, code bytes [16g, 16g+16) -> dims [32g, 32g+32)
      uint2 vw[4][2];
      uint32_t vsc;     // V scale bytes of group g for those rows
      {
        uint32_t sbytes[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t rb = slot + (16 * h + 2 * c + (j & 1) + 8 * (j >> 1)) * CONTENT;
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
          const int tok = t0 + 16 * h + 2 * c + (j & 1) + 8 * (j >> 1);
          if (tok >= L) {
            vw[j][0] = make_uint2(0, 0);
            vw[j][1] = make_uint2(0, 0);
            vsc &= ~(0xffu << (8 * j));
          }
        }
      }
      // {s[2c], s[2c+1]} and {s[2c+8], s[2c+9]}; a zeroed byte is 0 in both formats
      const uint32_t vs01 = ue8m0 ? ue8m0x2_lo_to_f16x2(vsc) : e4m3x2_lo_to_f16x2(vsc);
      const uint32_t vs89 = ue8m0 ? ue8m0x2_lo_to_f16x2(vsc >> 16) : e4m3x2_hi_to_f16x2(vsc);
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
            fa[bq][0] = lds32(lut + (((Ea >> (8 * bq)) & 0xFFu) * (LUT_COPIES * 4)));
            fa[bq][1] = lds32(lut + (((Oa >> (8 * bq)) & 0xFFu) * (LUT_COPIES * 4)));
            fa[bq][2] = lds32(lut + (((Eb >> (8 * bq)) & 0xFFu) * (LUT_COPIES * 4)));
            fa[bq][3] = lds32(lut + (((Ob >> (8 * bq)) & 0xFFu) * (LUT_COPIES * 4)));
          }
        }
#pragma unroll
        for (int bq = 0; bq < 4; ++bq) {
          const int i = 4 * wq + bq;
          mma_f16_16816(o[i], hmul2(fa[bq][0], vs01), hmul2(fa[bq][1], vs01), hmul2(fa[bq][2], vs89),
                        hmul2(fa[bq][3], vs89), bP[h][0], bP[h][1]);
        }
      }
    }
    __syncwarp();
  }
}

// Combine the partitions of one query row (combine_row) and rotate it back:
// out = o_r H/16, 8 butterfly stages over the 256 dims (128 pairs per stage,
// one or two per thread: a row CTA has at least 64 threads).
template <typename OutT>
__global__ void __launch_bounds__(kCombineMaxThreads)
uq_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_m,
                  const float* __restrict__ part_l, OutT* __restrict__ out, int num_kv_heads, int qg,
                  int num_partitions, long long out_stride_seq, long long out_stride_head, int rot_perm) {
  constexpr int D = 256;
  extern __shared__ __align__(16) float sw[];
  __shared__ __align__(16) float vec[D];
  pdl_wait_primary();
  const int row = blockIdx.x;
  const int r = row % qg;
  const int sk = row / qg;
  const int seq = sk / num_kv_heads, kvh = sk % num_kv_heads;
  const int tid = threadIdx.x;
  combine_row<D, kCombineKmax256>(part_o, part_m, part_l, (long long)sk * num_partitions * qg + r, qg,
                                  num_partitions, sw, vec);
  const int pa = tid, pb = tid + blockDim.x;      // this thread's pairs (pb only when blockDim is 64)
  for (int st = 1; st < D; st <<= 1) {
    const int ia = ((pa & ~(st - 1)) << 1) | (pa & (st - 1));   // index with bit `st` clear
    const int ib = ((pb & ~(st - 1)) << 1) | (pb & (st - 1));
    float xa = 0.f, ya = 0.f, xb = 0.f, yb = 0.f;
    if (pa < D / 2) { xa = vec[ia]; ya = vec[ia + st]; }
    if (pb < D / 2) { xb = vec[ib]; yb = vec[ib + st]; }
    __syncthreads();
    if (pa < D / 2) { vec[ia] = xa + ya; vec[ia + st] = xa - ya; }
    if (pb < D / 2) { vec[ib] = xb + yb; vec[ib + st] = xb - yb; }
    __syncthreads();
  }
  if (tid < D / 4) {
    // with the column-permuted rotation M, out[i] = (o_r H / 16)[perm(i)]
    // (perm keeps bits 0..3, so four consecutive dims stay together)
    const int src = rot_perm ? rot_perm_dest(4 * tid) : 4 * tid;
    OutT* dst = out + seq * out_stride_seq + (long long)(kvh * qg + r) * out_stride_head + 4 * tid;
    store4(dst, vec[src] * 0.0625f, vec[src + 1] * 0.0625f, vec[src + 2] * 0.0625f, vec[src + 3] * 0.0625f);
  }
}

// ------------------------------------------------------------------ host side
// Warps per item: the smallest W (fewest merges) among those that minimise the
// per-warp slice count of the launch, rounds x slices per warp per item, with
// items bounded by the longest sequence the block table allows.
int uq_warps_per_item(long long items, int max_blocks, int block_size, int num_partitions, int num_sms) {
  const long long groups_per_tile = (long long)uq::TG / uq::SLICE;
  const long long tiles = ((long long)max_blocks * block_size + uq::TG - 1) / uq::TG;
  const long long tiles_per_item = std::max<long long>(1, (tiles + num_partitions - 1) / num_partitions);
  int best_w = 4;
  long long best = -1;
  for (int w = 1; w <= 4; w *= 2) {
    const long long slots = (long long)uq::CTAS_PER_SM * num_sms * (uq::NW / w);
    const long long rounds = (items + slots - 1) / slots;
    const long long cost = rounds * tiles_per_item * groups_per_tile / w;
    if (best < 0 || cost < best) { best = cost; best_w = w; }
  }
  return best_w;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (no
// link-time dependency on the driver library); null if the driver lacks it.
static EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

cudaError_t launch_uq_partition(const UqLaunch& a, cudaStream_t stream) {
  // the slot cache as a 3-D tensor of 2-byte units: x = unit within a
  // (token, head) slot, y = KV head, z = token row (block * block_size + t);
  // a box is 136 units (the 272 used bytes) x 1 head x 16 token rows
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap kv_map;
  const cuuint64_t dims[3] = {(cuuint64_t)(a.padded_slot / 2), (cuuint64_t)a.num_kv_heads,
                              (cuuint64_t)a.num_blocks * (cuuint64_t)a.block_size};
  const cuuint64_t strides[2] = {(cuuint64_t)a.padded_slot, (cuuint64_t)a.padded_slot * a.num_kv_heads};
  const cuuint32_t box[3] = {uq::CONTENT / 2, 1, uq::TMA_ROWS};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(&kv_map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint8_t*>(a.kv), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
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
  p.flags = a.flags;
  const long long items = (long long)a.num_seqs * a.num_kv_heads * a.num_partitions;
  if (items <= 0) return cudaSuccess;
  const int W = uq_warps_per_item(items, a.max_blocks, a.block_size, a.num_partitions, a.num_sms);
  const long long ctas = (items + uq::NW / W - 1) / (uq::NW / W);
  const int grid = (int)std::min<long long>(ctas, (long long)uq::CTAS_PER_SM * a.num_sms);
  auto launch = [&](auto kern) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, uq::SMEM);
    kern<<<grid, uq::THREADS, uq::SMEM, stream>>>(kv_map, p);
  };
  if (W == 1) launch(uq_partition_kernel<1>);
  else if (W == 2) launch(uq_partition_kernel<2>);
  else launch(uq_partition_kernel<4>);
  return cudaGetLastError();
}

template <typename OutT>
static cudaError_t launch_uq_combine_t(const CombineLaunch& a, OutT* out, cudaStream_t stream) {
  const int grid = a.num_seqs * a.num_kv_heads * a.qg;
  const int threads = combine_threads(256, kCombineKmax256, a.num_partitions);
  const size_t smem = combine_smem_bytes(a.num_partitions, threads);
  if (smem > 40 * 1024)
    cudaFuncSetAttribute(uq_combine_kernel<OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, uq_combine_kernel<OutT>, a.part_o, a.part_m, a.part_l, out, a.num_kv_heads,
                            a.qg, a.num_partitions, a.out_stride_seq, a.out_stride_head, a.rot_perm);
}

cudaError_t launch_uq_combine(const CombineLaunch& a, cudaStream_t stream) {
  if (a.num_seqs * a.num_kv_heads * a.qg <= 0) return cudaSuccess;
  cudaError_t e = a.out_bf16 ? launch_uq_combine_t(a, static_cast<__nv_bfloat16*>(a.out), stream)
                             : launch_uq_combine_t(a, static_cast<float*>(a.out), stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qpa
