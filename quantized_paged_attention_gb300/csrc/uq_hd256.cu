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
//  * a split of each sequence over partitions (STEP F strides 256-token tile
//    groups; here the stride granule is the 32-token slice, see below),
//    softmax partials (O, m, l) per (seq, kv_head, partition) (STEP G);
//  * the combine merges partitions and rotates the output back (o = o_r H/16).
// Readings: the group scales are e4m3 and V decodes through a 16-entry fp32
// centroid table (V = centroid[code] * scale); the page's own V convert
// (e2m1 * scale) is the case where the table is the e2m1 value table.
// Descriptor flags select the page's own formats: UE8M0 group scales
// (2^(byte-127)), the e4m3 rounding of softmax_scale * q_r after the rotation
// (the logits then take no further scale), and the rotation's column
// permutation (a permuted q load here, a permuted store in the combine).
//
// GB300 design. One persistent CTA per SM: two producer warps stream 32-token
// slices of a group of HG KV heads into a ring of shared-memory stages,
// alternate stages each (one tensor-map box of 32 token rows x 272 bytes per
// head, completion counted on the stage's mbarrier), and eight consumer warps
// compute. A work item is (sequence, head group, partition p), p owning the
// slices p, p+P, ... of the sequence (a sequence of 75000 tokens has 293
// tile groups, which no partition count divides evenly: strided slices keep
// the partitions within one slice of each other); consumer warp w
// owns one (head of the group, 8-row half of the query group) and every J-th
// slice of the item (J = 8 / (HG x halves)), keeps its own softmax state and
// writes it as its own partial slot, so the combine merges P x J slots per
// query row and no warp ever waits on another consumer. Per 16-token tile:
//  * K by ldmatrix: lane (g, c) receives word c of each 32-dim group's codes
//    for token rows g and g+8, so every f16 m16n8k16 MMA (e2m1 -> f16 with
//    cvt, exact) stays inside one scale group; the group's scale multiplies
//    the f32 partial dot afterwards (exact for e4m3 and for every UE8M0 byte);
//  * the query is rotated in registers (in-thread butterflies over dim bits
//    0..2 and 5..7, lane exchanges over bits 3..4, in stride order 1..128);
//  * V^T fragments built per token pair: the two tokens' nibbles of a dim form
//    one byte that is converted with cvt e2m1x2 (e2m1 table) or looked up in a
//    256-entry f16x2 table of centroid pairs normalised to |c| < 1 (16 bank
//    copies), times the token pair's scale in f16;
//  * with UE8M0 scales every token's V scales are split into its largest
//    power of two E_t and the rest (2^(b - E_t) <= 1, applied in f16); 2^E_t
//    enters the probability operand relative to a running reference exponent
//    R of the item, and 2^(R - 127) multiplies the output.
#include <cmath>

#include "qpa.h"
#include "common.cuh"
#include "qpa_internal.h"
#include "combine.cuh"
#include "tc.cuh"

namespace qpa {

namespace uq {
constexpr int D = 256;
constexpr int SLICE = 32;                        // tokens per stage: two 16-token MMA tiles
constexpr int NC = 8;                            // consumer warps
constexpr int NPW = 2;                           // producer warps (alternate stages)
constexpr int THREADS = (NC + NPW) * 32;
constexpr int CONTENT = 272;                     // used bytes of a slot
constexpr int HEAD_SLICE = SLICE * CONTENT;      // 8704: 32 slots of one head, dense
constexpr int KS_OFF = 128, VC_OFF = 136, VS_OFF = 264;
constexpr int LUT_COPIES = 16;                   // bank copies of each table entry
constexpr int LUT_BYTES = 256 * LUT_COPIES * 4;  // [code pair][bank copy] f16x2
constexpr int QF_BYTES = NC * 32 * 32 * 4;       // rotated query fragments: [warp][G][lane] x 16 B
constexpr int MAX_DEPTH = 12;
constexpr int SMEM_LIMIT = 232448;
constexpr int TAIL_BYTES = 2 * MAX_DEPTH * 8 + 16 + 128;   // barriers, abort flag, alignment slack
static_assert(HEAD_SLICE % 128 == 0, "stage alignment");
}  // namespace uq

struct UqParams {
  const uint16_t* q;
  const float* centroids;
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* part_o;
  float* part_m;
  float* part_l;
  long long q_stride_seq, q_stride_head;
  int num_seqs, num_kv_heads, qg, block_size, log2_bs, num_blocks, max_blocks, num_partitions;
  int hg, nh, jw, depth;   // heads per item, 8-row halves, slices per warp stride, ring stages
  float softmax_scale;
  int flags;               // QPA_UQ_Q_HAIRCUT | QPA_UQ_ROT_PERM (the scale format is the template)
};

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

// Number of 32-token slices of partition p (slices p, p+P, ... below L).
__device__ __forceinline__ int uq_slices(int L, int p, int P) {
  const int ns = (L + uq::SLICE - 1) / uq::SLICE;
  return p < ns ? (ns - 1 - p) / P + 1 : 0;
}

// Largest byte of the eight in w (lo, hi).
__device__ __forceinline__ uint32_t max_byte8(uint2 w) {
  uint32_t m = __vmaxu4(w.x, w.y);
  m = __vmaxu4(m, m >> 16);
  m = __vmaxu4(m, m >> 8);
  return m & 0xffu;
}
// 2^(b - e) as float32 for UE8M0 bytes b <= e; 0 for b = 0 (or b - e < -126).
__device__ __forceinline__ float pow2_diff(uint32_t b, uint32_t e) {
  const int t = (int)b - (int)e + 127;
  return (b == 0u || t <= 0) ? 0.f : __uint_as_float((uint32_t)t << 23);
}

template <bool UE8>
__global__ void __launch_bounds__(uq::THREADS, 1)
uq_partition_kernel(const __grid_constant__ CUtensorMap kv_map, const UqParams p) {
  using namespace uq;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the tensor-map copies need 128-byte aligned destinations
  uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int depth = p.depth;
  const int stage_bytes = p.hg * HEAD_SLICE;
  uint8_t* lut_p = smem + depth * stage_bytes;
  uint8_t* qf_p = lut_p + LUT_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(qf_p + QF_BYTES);
  uint64_t* empty = full + depth;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + depth);
  const int C = p.hg * p.nh;      // consumer warps per slice
  const int J = p.jw;             // = NC / C
  if (threadIdx.x == 0) {
    for (int i = 0; i < depth; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], C);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == NC * 32) prefetch_tmap(&kv_map);
  const int P = p.num_partitions;
  const int NHG = p.num_kv_heads / p.hg;
  const int num_items = p.num_seqs * NHG * P;
  const int bs = p.block_size;
  const int lbs = p.log2_bs;
  __syncthreads();   // the barriers are initialised

  const uint32_t ring = smem_u32(smem);
  auto item_len = [&](int item) -> int {
    const int seq = item / (NHG * P);
    return max(0, min(__ldg(p.seq_lens + seq), p.max_blocks * bs));
  };

  if (warp >= NC) {
    // ================================================================ producer
    // Two producer warps take alternate stages (one issuing thread streams
    // only about 36 GB/s of tensor-map boxes from HBM; an SM needs ~45). The
    // copy coordinates of an item's slices are computed 32 slices at a time,
    // lane l taking slice 32 c + l (its block-table entries loaded in
    // parallel, one chunk ahead); the per-stage path is then two shuffles,
    // the stage's empty wait by lane 0, and lane 0's copies.
    const int pw = warp - NC;
    const uint64_t pol = policy_evict_first();
    const bool two_boxes = bs < SLICE;   // block size 16: a slice spans two blocks
    int g = 0;                           // stages of the CTA so far (both warps count all)
    bool ok = true;
    for (int item = blockIdx.x; item < num_items && ok; item += gridDim.x) {
      const int seq = item / (NHG * P);
      const int rem = item % (NHG * P);
      const int part = rem / NHG, hgi = rem % NHG;
      const int L = item_len(item);
      const int32_t* bt = p.block_table + (long long)seq * p.max_blocks;
      // the table entries of slice k's first (and, block size 16, second) box:
      // they depend on the slice alone, so they are read while the sequence
      // length is still on its way, and masked by it afterwards
      auto entries = [&](int k, int& ra, int& rb) {
        const int t0 = (part + P * k) * SLICE;
        const int ea = t0 >> lbs, eb = (t0 + 16) >> lbs;
        ra = ea < p.max_blocks ? __ldg(bt + ea) : 0;
        rb = two_boxes && eb < p.max_blocks ? __ldg(bt + eb) : 0;
      };
      int ra, rb, rna, rnb;
      entries(lane, ra, rb);
      entries(32 + lane, rna, rnb);
      const int nsl = uq_slices(L, part, P);
      if (nsl == 0) continue;
      // token-row coordinates of slice k's first (and second) box from its entries
      auto coords = [&](int k, int ra, int rb, int& za, int& zb) {
        za = 0;
        zb = 0;
        if (k >= nsl) return;
        const int t0 = (part + P * k) * SLICE;
        int pa = ((t0 >> lbs) << lbs) < L ? ra : 0;
        if (pa < 0 || pa >= p.num_blocks) {
          atomicExch(&g_kernel_error, KERR_BAD_BLOCK);
          pa = 0;
        }
        if (!two_boxes) {
          za = pa * bs + (t0 & (bs - 1));
        } else {
          int pb = (((t0 + 16) >> lbs) << lbs) < L ? rb : 0;
          if (pb < 0 || pb >= p.num_blocks) {
            atomicExch(&g_kernel_error, KERR_BAD_BLOCK);
            pb = 0;
          }
          za = pa * bs;
          zb = pb * bs;
        }
      };
      // the current chunk's coordinates; the next chunk's table entries are
      // read one chunk ahead and turned into coordinates only when it starts
      int za, zb;
      coords(lane, ra, rb, za, zb);
      int chunk = 0;
      const uint32_t head0 = hgi * p.hg;
      // this warp's slices: stage g + k with (g + k) % NPW == pw
      for (int k = (pw - g % NPW + NPW) % NPW; k < nsl; k += NPW) {
        if ((k >> 5) != chunk) {
          chunk = k >> 5;
          coords(32 * chunk + lane, rna, rnb, za, zb);
          entries(32 * (chunk + 1) + lane, rna, rnb);
        }
        const int ya = __shfl_sync(0xffffffffu, za, k & 31);
        const int yb = __shfl_sync(0xffffffffu, zb, k & 31);
        const int gs = g + k;
        const int s = gs % depth;
        const uint32_t eph = ((uint32_t)(gs / depth) & 1u) ^ 1u;   // a fresh barrier passes parity 1
        if (lane == 0) {
          if (!mbar_try_wait(&empty[s], eph)) ok = role_wait(&empty[s], eph, abort_flag, KERR_TIMEOUT_EMPTY);
          if (ok) {
            // every head's 32 token slots, 272 bytes each, land densely in the
            // stage; slots past the end of the sequence are read from the blocks
            // the table names (or block 0) and masked by the consumers
            mbar_arrive_expect_tx(&full[s], stage_bytes);
            uint32_t dst = ring + s * stage_bytes;
            for (int hh = 0; hh < p.hg; ++hh, dst += HEAD_SLICE) {
              tma_load_3d(dst, &kv_map, 0, head0 + hh, ya, &full[s], pol);
              if (two_boxes) tma_load_3d(dst + 16 * CONTENT, &kv_map, 0, head0 + hh, yb, &full[s], pol);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      g += nsl;
    }
    // give the copies still in flight a bounded time to land before the CTA's
    // shared memory goes away (they complete whether or not anyone consumes them)
    for (int i = max(0, g - depth); i < g; ++i) mbar_wait(&full[i % depth], (uint32_t)(i / depth) & 1u, KERR_TIMEOUT_FULL);
    return;
  }

  // ================================================================== consumers
  // ---- centroid table (consumer warps: the producers started streaming
  // without it): the e2m1 table takes the cvt path, anything else the
  // shared-memory pair table of the centroids divided by 2^cexp (|c| < 1, so
  // no f16 product with a scale overflows); the output is multiplied back.
  bool e2m1_table = true;
  int cexp = 0;
  {
    float cv[16];
    float cmax = 0.f;
    bool finite = true;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      cv[k] = __ldg(p.centroids + k);
      e2m1_table = e2m1_table && (cv[k] == e2m1_value(k)) && (__float_as_uint(cv[k]) >> 31) == (uint32_t)(k >> 3);
      finite = finite && isfinite(cv[k]);
      cmax = fmaxf(cmax, fabsf(cv[k]));
    }
    if (!finite && threadIdx.x == 0) atomicExch(&g_kernel_error, KERR_RANGE);
    if (!e2m1_table) {
      if (cmax > 0.f && finite) frexpf(cmax, &cexp);
      uint32_t* t = reinterpret_cast<uint32_t*>(lut_p);
      for (int i = threadIdx.x; i < 256 * LUT_COPIES; i += NC * 32) {
        const int e = i / LUT_COPIES;
        t[i] = f32x2_to_f16x2(ldexpf(cv[e & 15], -cexp), ldexpf(cv[e >> 4], -cexp));
      }
    }
  }
  named_barrier(1, NC * 32);   // the table is built (the consumer warps alone)

  const int cw = warp % C, jr = warp / C;
  const int hh = cw / p.nh, hf = cw % p.nh;
  const int g = lane >> 2;
  const int c = lane & 3;
  const bool haircut = (p.flags & QPA_UQ_Q_HAIRCUT) != 0;
  const bool rot_perm = (p.flags & QPA_UQ_ROT_PERM) != 0;
  // with the haircut the softmax scale is already inside the e4m3 query
  const float rowc = haircut ? kLog2e : p.softmax_scale * kLog2e;
  const uint32_t lut = smem_u32(lut_p) + (lane & (LUT_COPIES - 1)) * 4;   // this lane's bank copy
  // ldmatrix row addresses of K codes: lane l feeds matrix l/8 (rows 0..7 or
  // 8..15 of a tile, group 2m or 2m+1), row l%8
  const uint32_t k_lane_off = (uint32_t)(((lane & 7) + ((lane >> 3) & 1) * 8) * CONTENT + 16 * (lane >> 4));
  const long long slots_per_head = (long long)P * J;

  int gbase = 0;
  for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
    const int seq = item / (NHG * P);
    const int rem = item % (NHG * P);
    const int part = rem / NHG, hgi = rem % NHG;
    const int L = item_len(item);
    const int nsl = uq_slices(L, part, P);
    const int head = hgi * p.hg + hh;
    // this warp's partial slot: rows r of (seq, head, slot part * J + jr)
    const long long row0 = (((long long)seq * p.num_kv_heads + head) * slots_per_head + (long long)part * J + jr) * p.qg;
    if (nsl <= jr) {
      // no slice of this item is this warp's: an empty slot (O is never read)
      if (lane < 8 && 8 * hf + lane < p.qg) {
        p.part_m[row0 + 8 * hf + lane] = -INFINITY;
        p.part_l[row0 + 8 * hf + lane] = 0.f;
      }
      gbase += nsl;
      continue;
    }

    // ---- rotated query: row 8 hf + g, dims {32 G + 8 c + e}; butterflies over
    // dim bits 0..2 (in-thread), 3..4 (lanes c^1, c^2) and 5..7 (in-thread), in
    // stride order 1, 2, ..., 128. With the column-permuted rotation, position
    // m takes q[perm^-1(m)] (the permutation moves index bits 4..6 only, so it
    // commutes through the Hadamard and 8-dim runs stay contiguous).
    // this warp's fragments: group G's four f16x2 words of lane l at (G * 32 + l) * 16
    const uint32_t qfrag = smem_u32(qf_p) + warp * (32 * 32 * 4) + lane * 16;
    {
      float v[64];
      const int qrow = 8 * hf + g;
      if (qrow < p.qg) {
        const uint16_t* qsrc = p.q + (long long)seq * p.q_stride_seq + (long long)(head * p.qg + qrow) * p.q_stride_head;
#pragma unroll
        for (int G = 0; G < 8; ++G) {
          const int m = 32 * G + 8 * c;
          const int src = rot_perm ? rot_perm_source(m) : m;
          const uint4 w4 = __ldg(reinterpret_cast<const uint4*>(qsrc + src));
          const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            v[8 * G + 2 * k] = __uint_as_float(ws[k] << 16);
            v[8 * G + 2 * k + 1] = __uint_as_float(ws[k] & 0xffff0000u);
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < 64; ++k) v[k] = 0.f;
      }
#pragma unroll
      for (int st = 1; st < 8; st <<= 1) {          // dim bits 0..2
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if ((k & st) == 0) {
            const float x = v[k], y = v[k + st];
            v[k] = x + y;
            v[k + st] = x - y;
          }
      }
#pragma unroll
      for (int sh = 1; sh <= 2; sh <<= 1) {          // dim bits 3..4
        const bool upper = (c & sh) != 0;
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          const float pv = __shfl_xor_sync(0xffffffffu, v[k], sh);
          v[k] = upper ? pv - v[k] : v[k] + pv;
        }
      }
#pragma unroll
      for (int st = 8; st < 64; st <<= 1) {         // dim bits 5..7
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if ((k & st) == 0) {
            const float x = v[k], y = v[k + st];
            v[k] = x + y;
            v[k + st] = x - y;
          }
      }
      uint32_t qf[32];
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
#pragma unroll
      for (int G = 0; G < 8; ++G)
        sts_i4(qfrag + G * 512, make_int4(qf[4 * G], qf[4 * G + 1], qf[4 * G + 2], qf[4 * G + 3]));
      __syncwarp();
    }

    float o[16][4];           // O^T: m-tile i rows g, g+8 = dims 32g+2i, 32g+2i+1; cols rows 2c, 2c+1
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    int R = 0;                // UE8M0: the item's reference V exponent so far
    bool range_bad = false;
#pragma unroll
    for (int i = 0; i < 16; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[i][k] = 0.f;

    bool aborted = false;
    // stage of slice k: (gbase + k) % depth and its phase, kept incrementally
    // (J < depth)
    int s = (gbase + jr) % depth;
    uint32_t fph = (uint32_t)((gbase + jr) / depth) & 1u;
#pragma unroll 1
    for (int k = jr; k < nsl; k += J) {
      if (k > jr && (s += J) >= depth) {
        s -= depth;
        fph ^= 1u;
      }
      if (!warp_wait(&full[s], fph, abort_flag, KERR_TIMEOUT_FULL)) {
        aborted = true;
        break;
      }
      const uint32_t slot = ring + s * stage_bytes + hh * HEAD_SLICE;
      const int t0 = (part + P * k) * SLICE;
      const bool partial = t0 + SLICE > L;

      // ---- S^T (16 tokens x 8 rows) = K q_r^T per tile, one 32-dim scale
      // group at a time; the group's scale multiplies its f32 partial dot
      float x[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint2 sca = lds64(slot + (16 * h + g) * CONTENT + KS_OFF);
        const uint2 scb = lds64(slot + (16 * h + g + 8) * CONTENT + KS_OFF);
        float xa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          // word c of the codes of groups 2m, 2m+1 for token rows g, g+8
          uint32_t kg[2], kg8[2];
          ldsm_x4(slot + 16 * h * CONTENT + k_lane_off + 32 * m, kg[0], kg8[0], kg[1], kg8[1]);
          // scales of groups 2m, 2m+1 for rows g, g+8
          const uint32_t wa = (m < 2 ? sca.x : sca.y) >> (16 * (m & 1));
          const uint32_t wb = (m < 2 ? scb.x : scb.y) >> (16 * (m & 1));
          float ska[2], skb[2];
          if constexpr (UE8) {
            ska[0] = __uint_as_float((wa & 0xffu) << 23);          // 2^(b-127), b = 0 -> 0
            ska[1] = __uint_as_float(((wa >> 8) & 0xffu) << 23);
            skb[0] = __uint_as_float((wb & 0xffu) << 23);
            skb[1] = __uint_as_float(((wb >> 8) & 0xffu) << 23);
          } else {
            const uint32_t a2 = e4m3x2_lo_to_f16x2(wa), b2 = e4m3x2_lo_to_f16x2(wb);
            ska[0] = f16_lo_to_f32(a2); ska[1] = f16_hi_to_f32(a2);
            skb[0] = f16_lo_to_f32(b2); skb[1] = f16_hi_to_f32(b2);
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int G = 2 * m + u;
            const int4 qg4 = lds_i4(qfrag + G * 512);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            // k-slots 2c, 2c+1 | 2c+8, 2c+9 hold dims 32G + 8c + 4h' + {0,1} | {2,3}
            mma_f16_16816(acc, e2m1x2_to_f16x2<0>(kg[u]), e2m1x2_to_f16x2<0>(kg8[u]), e2m1x2_to_f16x2<1>(kg[u]),
                          e2m1x2_to_f16x2<1>(kg8[u]), (uint32_t)qg4.x, (uint32_t)qg4.y);
            mma_f16_16816(acc, e2m1x2_to_f16x2<2>(kg[u]), e2m1x2_to_f16x2<2>(kg8[u]), e2m1x2_to_f16x2<3>(kg[u]),
                          e2m1x2_to_f16x2<3>(kg8[u]), (uint32_t)qg4.z, (uint32_t)qg4.w);
            xa[0] = fmaf(ska[u], acc[0], xa[0]);
            xa[1] = fmaf(ska[u], acc[1], xa[1]);
            xa[2] = fmaf(skb[u], acc[2], xa[2]);
            xa[3] = fmaf(skb[u], acc[3], xa[3]);
          }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) x[h][r] = xa[r] * rowc;
        const bool va = !partial || t0 + 16 * h + g < L, vb = !partial || t0 + 16 * h + g + 8 < L;
        if constexpr (UE8) {
          // a scale byte of 255 (not a power of two the format defines) or a
          // logit beyond float32 range
          range_bad = range_bad || (va && !(isfinite(x[h][0]) && isfinite(x[h][1]))) ||
                      (vb && !(isfinite(x[h][2]) && isfinite(x[h][3])));
        }
        if (!va) { x[h][0] = -INFINITY; x[h][1] = -INFINITY; }
        if (!vb) { x[h][2] = -INFINITY; x[h][3] = -INFINITY; }
      }

      // ---- UE8M0: the largest V scale byte of tokens g, g+8 of each tile
      // (0 past the end of the sequence) and the item's reference exponent
      uint32_t ev[2] = {0u, 0u};      // [tile]: E(token g) | E(token g+8) << 16
      int Rn = R;
      if constexpr (UE8) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t ea = (!partial || t0 + 16 * h + g < L) ? max_byte8(lds64(slot + (16 * h + g) * CONTENT + VS_OFF)) : 0u;
          const uint32_t eb = (!partial || t0 + 16 * h + g + 8 < L) ? max_byte8(lds64(slot + (16 * h + g + 8) * CONTENT + VS_OFF)) : 0u;
          ev[h] = ea | (eb << 16);
          Rn = max(Rn, (int)max(ea, eb));
        }
        Rn = (int)__reduce_max_sync(0xffffffffu, (unsigned)Rn);
        range_bad = range_bad || Rn == 255;
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
      if (__any_sync(0xffffffffu, (mn0 > m_run[0]) || (mn1 > m_run[1])) || Rn > R) {
        float a0 = ex2(m_run[0] - mn0), a1 = ex2(m_run[1] - mn1);
        l_run[0] *= a0;
        l_run[1] *= a1;
        if (UE8 && Rn > R) {
          const float fr = pow2_diff((uint32_t)R + 1u, (uint32_t)Rn + 1u);   // 2^(R - Rn), exact
          a0 *= fr;
          a1 *= fr;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          o[i][0] *= a0; o[i][1] *= a1;
          o[i][2] *= a0; o[i][3] *= a1;
        }
        m_run[0] = mn0;
        m_run[1] = mn1;
        R = Rn;
      }
      uint32_t bP[2][2];      // P^T B fragments per tile (tokens 2c.., 2c+8.. x row g)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t P01 = f32x2_to_f16x2(ex2(x[h][0] - mn0), ex2(x[h][1] - mn1));
        uint32_t P23 = f32x2_to_f16x2(ex2(x[h][2] - mn0), ex2(x[h][3] - mn1));
        l_run[0] += f16_lo_to_f32(P01) + f16_lo_to_f32(P23);
        l_run[1] += f16_hi_to_f32(P01) + f16_hi_to_f32(P23);
        if constexpr (UE8) {
          // the probability operand carries 2^(E_t - R) of its token
          const float fa = pow2_diff(ev[h] & 0xffffu, (uint32_t)R), fb = pow2_diff(ev[h] >> 16, (uint32_t)R);
          P01 = hmul2(P01, f32x2_to_f16x2(fa, fa));
          P23 = hmul2(P23, f32x2_to_f16x2(fb, fb));
        }
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
        uint32_t vs01, vs89;
        if constexpr (UE8) {
          // 2^(b - E_t): the token's largest power of two stays out of V
          const uint32_t e0 = __shfl_sync(0xffffffffu, ev[h], 8 * c);       // tokens 2c | 2c+8
          const uint32_t e1 = __shfl_sync(0xffffffffu, ev[h], 8 * c + 4);   // tokens 2c+1 | 2c+9
          vs01 = f32x2_to_f16x2(pow2_diff(vsc & 0xffu, e0 & 0xffffu), pow2_diff((vsc >> 8) & 0xffu, e1 & 0xffffu));
          vs89 = f32x2_to_f16x2(pow2_diff((vsc >> 16) & 0xffu, e0 >> 16), pow2_diff(vsc >> 24, e1 >> 16));
        } else {
          vs01 = e4m3x2_lo_to_f16x2(vsc);
          vs89 = e4m3x2_hi_to_f16x2(vsc);
        }
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
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (aborted) break;
    if (UE8 && __any_sync(0xffffffffu, range_bad) && lane == 0) atomicExch(&g_kernel_error, KERR_RANGE);

    // ---- this warp's softmax state is its slot's partial: normalise and write
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
      l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], sh);
      l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], sh);
    }
    const int oexp = cexp + (UE8 ? R - 127 : 0);   // 2^oexp undoes the table and V-exponent scaling
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = 8 * hf + 2 * c + hr;
      if (r < p.qg) {
        const float inv = l_run[hr] > 0.f ? 1.f / l_run[hr] : 0.f;
        float* dst = p.part_o + (row0 + r) * D + 32 * g;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          *reinterpret_cast<float2*>(dst + 2 * i) =
              make_float2(ldexpf(o[i][hr] * inv, oexp), ldexpf(o[i][2 + hr] * inv, oexp));
        if (g == 0) {
          p.part_m[row0 + r] = m_run[hr] == -INFINITY ? -INFINITY : m_run[hr] * kLn2;
          p.part_l[row0 + r] = l_run[hr];
        }
      }
    }
    gbase += nsl;
  }
}

// Combine the partition slots of one query row (combine_row) and rotate it
// back: out = o_r H/16, 8 butterfly stages over the 256 dims (128 pairs per
// stage, one or two per thread: a row CTA has at least 64 threads).
template <typename OutT>
__global__ void __launch_bounds__(kCombineMaxThreads)
uq_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_m,
                  const float* __restrict__ part_l, OutT* __restrict__ out, int num_kv_heads, int qg,
                  int num_partitions, long long out_stride_seq, long long out_stride_head, int rot_perm) {
  constexpr int D = 256;
  extern __shared__ __align__(16) float sw[];
  __shared__ __align__(16) float vec[D];
  const int row = blockIdx.x;
  const int r = row % qg;
  const int sk = row / qg;
  const int seq = sk / num_kv_heads, kvh = sk % num_kv_heads;
  const int tid = threadIdx.x;
  combine_row<D, kCombineKmax256, true>(part_o, part_m, part_l, (long long)sk * num_partitions * qg + r, qg,
                                        num_partitions, sw, vec, threadIdx.x, blockDim.x);
  // o = o_r H / 16 by one warp: lane l holds dims 8l .. 8l + 7, the butterflies
  // of index bits 0..2 in registers and of bits 3..7 across lanes, in stride
  // order 1, 2, ..., 128; the 1/16 first, so that no butterfly sum exceeds the
  // final output's bound (16 max |o_r|)
  if (tid >= 32) return;
  float x[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) x[j] = vec[8 * tid + j] * 0.0625f;
#pragma unroll
  for (int st = 1; st < 8; st <<= 1)
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (!(j & st)) {
        const float a = x[j], b = x[j + st];
        x[j] = a + b;
        x[j + st] = a - b;
      }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool hi = (tid & m) != 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float other = __shfl_xor_sync(0xffffffffu, x[j], m);
      x[j] = hi ? other - x[j] : x[j] + other;
    }
  }
  // with the column-permuted rotation M, out[i] = (o_r H / 16)[perm(i)]; perm
  // keeps bits 0..3, so this lane's 8 dims are the outputs from
  // rot_perm_source(8 l) on
  const int dst0 = rot_perm ? rot_perm_source(8 * tid) : 8 * tid;
  OutT* dst = out + seq * out_stride_seq + (long long)(kvh * qg + r) * out_stride_head + dst0;
  store4(dst, x[0], x[1], x[2], x[3]);
  store4(dst + 4, x[4], x[5], x[6], x[7]);
}

// ------------------------------------------------------------------ host side
// Heads per item (HG, the largest of 8, 4, 2, 1 that divides Hk with at most
// eight (head, 8-row half) pairs and a ring of at least J + 2 stages), the
// consumer warps' slice stride J = 8 / (HG x halves), and the ring depth.
UqPlan uq_plan(int num_kv_heads, int query_group) {
  UqPlan pl{};
  pl.nh = (query_group + 7) / 8;
  for (int hg = 8; hg >= 1; hg >>= 1) {
    if (num_kv_heads % hg || hg * pl.nh > uq::NC) continue;
    const int c = hg * pl.nh;
    const int j = uq::NC / c;
    const int stage = hg * uq::HEAD_SLICE;
    const int depth =
        std::min(uq::MAX_DEPTH, (uq::SMEM_LIMIT - uq::LUT_BYTES - uq::QF_BYTES - uq::TAIL_BYTES) / stage);
    if (depth < j + 2) continue;
    pl.hg = hg;
    pl.jw = j;
    pl.depth = depth;
    pl.smem = depth * stage + uq::LUT_BYTES + uq::QF_BYTES + uq::TAIL_BYTES;
    return pl;
  }
  return pl;   // hg = 0: not reachable for query_group <= 16 (hg = 1 always fits)
}

EncodeTiledFn encode_tiled() {
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
  // the slot cache as a 3-D tensor of 8-byte units: x = unit within a
  // (token, head) slot, y = KV head, z = token row (block * block_size + t);
  // a box is the 34 units of the 272 used bytes x 1 head x 32 token rows (16
  // for block size 16), landing as dense 272-byte rows
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  const UqPlan pl = uq_plan(a.num_kv_heads, a.qg);
  if (pl.hg == 0) return cudaErrorInvalidValue;
  CUtensorMap kv_map;
  const cuuint64_t dims[3] = {(cuuint64_t)(a.padded_slot / 8), (cuuint64_t)a.num_kv_heads,
                              (cuuint64_t)a.num_blocks * (cuuint64_t)a.block_size};
  const cuuint64_t strides[2] = {(cuuint64_t)a.padded_slot, (cuuint64_t)a.padded_slot * a.num_kv_heads};
  const cuuint32_t box[3] = {uq::CONTENT / 8, 1, (cuuint32_t)std::min(a.block_size, uq::SLICE)};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(&kv_map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint8_t*>(a.kv), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  UqParams p;
  p.q = static_cast<const uint16_t*>(a.q);
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
  p.hg = pl.hg;
  p.nh = pl.nh;
  p.jw = pl.jw;
  p.depth = pl.depth;
  p.softmax_scale = a.softmax_scale;
  p.flags = a.flags & (QPA_UQ_Q_HAIRCUT | QPA_UQ_ROT_PERM);
  const long long items = (long long)a.num_seqs * (a.num_kv_heads / pl.hg) * a.num_partitions;
  if (items <= 0) return cudaSuccess;
  const int grid = (int)std::min<long long>(items, (long long)a.num_sms);
  auto launch = [&](auto kern) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
    kern<<<grid, uq::THREADS, pl.smem, stream>>>(kv_map, p);
  };
  if (a.flags & QPA_UQ_UE8M0_SCALES) launch(uq_partition_kernel<true>);
  else launch(uq_partition_kernel<false>);
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
  // plain stream order: launched as a programmatic dependent of the partition
  // grid (its CTAs cannot sit beside the partition CTAs) the step took ~5 us more
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
