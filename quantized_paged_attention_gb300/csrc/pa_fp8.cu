// fp8 (e4m3fn, per-tensor scale) paged-attention decode: split-KV partition
// kernel and flash-combine kernel.
//
// What it computes follows the ROCm/FlyDSL PR #825 page ("perf(pa tile):
// readable tile-programming PA decode kernel": per-tensor fp8 K/V, query
// length 1, GQA, cross-CTA partition split and a parallel flash-combine
// reduce) and the partition map of the ultraquant_decode_hd256 page (STEP F:
// partition p owns the 256-token tile groups p, p+P, p+2P, ...).
//
// GB300 design (not the pages' AMD design):
//  * persistent CTAs of four warps, three per SM. Each CTA walks its work
//    items (seq, kv_head, partition); inside an item warp w owns the 16-token
//    slices 4k+w of every tile group, so each slice is one page chunk
//    (block_size 16) or a 16-row piece of one (larger blocks).
//  * every warp runs its own copy pipeline: 16-byte cp.async copies (L1
//    bypass, L2 evict-first) of each slice's K and V chunks, 4 events deep,
//    into a private shared-memory ring, XOR-swizzled so the fragment reads
//    below are conflict-free; the 8 copies of a slice use per-lane offsets
//    computed once and immediate displacements. Query rows travel in the
//    same event stream.
//    There is no producer warp and no cross-warp handshake on the stream;
//    the block table is read one tile group ahead.
//  * QK runs on f16 mma.sync (m16n8k16): K bytes are converted e4m3 -> f16
//    (exact) in registers; each bf16 query row is scaled by a power of two so
//    its largest element lands in [2^14, 2^15) and rounded to f16, which is
//    exact for every element within 2^23 of the row maximum. (fp8 mma.sync
//    on sm_103a is lowered to conversions plus f16 MMAs, about 11 issued
//    instructions each, so converting K once here is cheaper.)
//  * PV runs on f16 mma.sync (m16n8k16): V bytes are paired across tokens with
//    prmt and converted to f16 (exact), P is rounded to f16 and transposed
//    into the B operand with movmatrix;
//  * each warp keeps its own online-softmax state; at the end of an item the
//    four states are rescaled to the common maximum and summed in a fixed
//    order (deterministic) through each warp's just-consumed ring slot.
#include "common.cuh"
#include "qpa_internal.h"
#include "combine.cuh"

namespace qpa {

namespace fp8 {
constexpr int D = 128;          // head_dim
constexpr int TG = 256;         // tile-group tokens
constexpr int SLICE = 16;       // tokens per warp step (one mma M tile)
constexpr int NW = 4;           // warps per CTA
constexpr int THREADS = NW * 32;
constexpr int DEPTH = 4;        // ring slots per warp (DEPTH-1 copy events in flight)
constexpr int SLOT_BYTES = 4096;   // one slice (K 2 KB + V 2 KB) or one item's query rows

template <int NT>
struct Smem {
  static constexpr int ringOff = 0;
  static constexpr int ringBytes = NW * DEPTH * SLOT_BYTES;
  static constexpr int mOff = ringOff + ringBytes;                // [NW][8NT] f32 running max
  static constexpr int lOff = mOff + NW * 8 * NT * 4;             // [NW][8NT] f32 running sum
  static constexpr int fOff = lOff + NW * 8 * NT * 4;             // [NW] scratch-slot address
  static constexpr int total = fOff + NW * 4;
};
template <int NT>
constexpr int ctas_per_sm() { return NT == 1 ? 3 : 2; }
}  // namespace fp8

struct Fp8Params {
  const uint16_t* q;          // bf16 bits
  const uint8_t* kv;          // [NB][2][Hk][bs][128]
  const int32_t* block_table;
  const int32_t* seq_lens;
  const float* k_scale;
  const float* v_scale;
  float* part_o;              // [B][Hk][P][QG][D]
  float* part_m;              // [B][Hk][P][QG]
  float* part_l;              // [B][Hk][P][QG]
  long long q_stride_seq, q_stride_head;   // elements
  int num_seqs, num_kv_heads, qg, block_size, log2_bs, num_blocks, max_blocks, num_partitions;
  float softmax_scale;
};

enum : int { EV_NONE = 0, EV_ITEM = 1, EV_SLICE = 2 };

template <int NT>
__global__ void __launch_bounds__(fp8::THREADS, fp8::ctas_per_sm<NT>())
pa_fp8_partition_kernel(const Fp8Params p) {
  using namespace fp8;
  using S = Smem<NT>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_items = p.num_seqs * p.num_kv_heads * p.num_partitions;
  const int P = p.num_partitions;
  const int bs = p.block_size;
  const int lbs = p.log2_bs;
  const int bpt = TG / bs > 0 ? TG / bs : 1;      // table entries per tile group
  float* ms = reinterpret_cast<float*>(smem + S::mOff);
  float* ls = reinterpret_cast<float*>(smem + S::lOff);
  uint32_t* fslot = reinterpret_cast<uint32_t*>(smem + S::fOff);
  pdl_launch_dependents();   // the combine kernel waits for this grid before reading

  const uint64_t pol = policy_evict_first();
  const uint32_t ring = smem_u32(smem + S::ringOff) + warp * DEPTH * SLOT_BYTES;
  const size_t head_bytes = size_t(bs) * D;                     // one (block, K/V, head) chunk
  const size_t v_off = size_t(p.num_kv_heads) * head_bytes;     // K chunk -> V chunk

  // ---------------------------------------------------------------- issue side
  // The warp walks its own event stream: for every item of this CTA, an item
  // event (copies the item's query rows) followed by the item's slices owned
  // by this warp (slice 4k + warp of every tile group). Events are issued
  // DEPTH-1 ahead of their use; lane (e % DEPTH) keeps event e's record.
  int ik_item = blockIdx.x;       // global index of the issue cursor's item
  int i_state = 0;                // 0: item event next, 1: slices next
  int i_tg = 0, i_kk = 0;
  int i_L = 0, i_Lnext = 0;
  int i_seq = 0, i_kvh = 0, i_part = 0;
  int32_t i_ent = 0, i_nent = 0;  // table entries of the current / next tile group (lane j: entry j)
  size_t kvh_off = 0;              // byte offset of the KV head's chunk inside a block
  int rec_a = 0, rec_b = 0;        // event record: (payload << 2) | kind, length
  // per-lane constants of the slice copies (see cp_async_chunk_pair)
  const int l3 = lane >> 3, j8 = lane & 7;
  const uint32_t doff0 = l3 * D + ((j8 ^ l3) << 4);
  const uint32_t doff1 = l3 * D + ((j8 ^ (l3 | 4)) << 4);
  const uint32_t l16 = lane * 16;
  const size_t blk_bytes = size_t(2) * p.num_kv_heads * head_bytes;   // one block: K and V of all heads

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
    int kind = EV_NONE, a = 0, b = 0;
    while (true) {
      if (ik_item >= num_items) break;
      if (i_state == 0) {
        i_part = ik_item % P;
        const int t = ik_item / P;
        i_kvh = t % p.num_kv_heads;
        i_seq = t / p.num_kv_heads;
        kvh_off = size_t(i_kvh) * head_bytes;
        if (i_part * TG < i_L) {
          // query rows of (seq, kv_head): qg rows x 256 B, 16 B per copy
          const uint16_t* qrow0 = p.q + i_seq * p.q_stride_seq + (long long)(i_kvh * p.qg) * p.q_stride_head;
          for (int idx = lane; idx < p.qg * 16; idx += 32) {
            const int row = idx >> 4, ch = idx & 15;
            cp_async16(slot + row * 256 + ch * 16, qrow0 + row * p.q_stride_head + ch * 8, pol);
          }
          i_ent = load_entries(i_seq, i_part, i_L);
          if ((i_part + P) * TG < i_L) i_nent = load_entries(i_seq, i_part + P, i_L);
        }
        i_state = 1;
        i_tg = i_part;
        i_kk = 0;
        kind = EV_ITEM; a = ik_item; b = i_L;
        break;
      }
      if (i_tg * TG >= i_L) {          // item exhausted: move to the CTA's next item
        ik_item += gridDim.x;
        i_state = 0;
        i_L = i_Lnext;
        i_Lnext = load_len(ik_item + gridDim.x);
        continue;
      }
      const int s = (i_tg * TG) / SLICE + 4 * i_kk + warp;   // 16-token slice index in the sequence
      const bool valid = s * SLICE < i_L;
      int phys = __shfl_sync(0xffffffffu, i_ent, ((s * SLICE) & (TG - 1)) >> lbs);
      if (++i_kk == 4) {               // next tile group of this item
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
      const uint8_t* kb = p.kv + size_t(phys) * blk_bytes + kvh_off + size_t((s * SLICE) & (bs - 1)) * D + l16;
      cp_async_chunk_pair(slot + doff0, slot + doff1, kb, kb + v_off, pol);
      kind = EV_SLICE; a = s; b = i_L;
      break;
    }
    cp_async_commit();
    if (lane == e % DEPTH) { rec_a = (a << 2) | kind; rec_b = b; }
  };

  // ---------------------------------------------------------------- consume side
  const int g = lane >> 2;      // fragment group id (row within 8)
  const int c = lane & 3;       // thread within group
  const float kscale = __ldg(p.k_scale);
  const float vscale = __ldg(p.v_scale);
  const float base_scale = kscale * p.softmax_scale * kLog2e;

  uint32_t qf[NT][16];   // query row 8nt+g, dims [32c, 32c+32), scaled, f16x2
  float rowc[NT][2];
  float o[NT][8][4];
  float m_run[NT][2], l_run[NT][2];
  int cur_item = -1;

  // Event e lives in slot e % DEPTH. Iteration e first refills the slot that
  // iteration e-1 read (all lanes are past those reads: every iteration ends
  // with __syncwarp), so DEPTH-1 events stay in flight while event e is
  // computed. At an item boundary that slot, not yet refilled, is this warp's
  // scratch for the merge.
#pragma unroll 1
  for (int e = 0; e < DEPTH - 1; ++e) issue(e);

#pragma unroll 1
  for (int e = 0;; ++e) {
    const int ra = __shfl_sync(0xffffffffu, rec_a, e % DEPTH);
    const int eb = __shfl_sync(0xffffffffu, rec_b, e % DEPTH);
    const int kind = ra & 3, ea = ra >> 2;

    if (kind != EV_SLICE && cur_item >= 0) {
      // ---- end of the current item: merge the four warps' (m, l, O) in a
      // fixed order and write this partition's partials.
      const long long row0 = (long long)cur_item * p.qg;     // item index = (seq*Hk + kvh)*P + part
      const uint32_t myfree = ring + ((e + DEPTH - 1) % DEPTH) * SLOT_BYTES;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
          l_run[nt][0] += __shfl_xor_sync(0xffffffffu, l_run[nt][0], sh);
          l_run[nt][1] += __shfl_xor_sync(0xffffffffu, l_run[nt][1], sh);
        }
        if (g == 0) {
          ms[warp * 8 * NT + nt * 8 + 2 * c] = m_run[nt][0];
          ms[warp * 8 * NT + nt * 8 + 2 * c + 1] = m_run[nt][1];
          ls[warp * 8 * NT + nt * 8 + 2 * c] = l_run[nt][0];
          ls[warp * 8 * NT + nt * 8 + 2 * c + 1] = l_run[nt][1];
        }
      }
      if (lane == 0) fslot[warp] = myfree;
      named_barrier(1, THREADS);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        // rescale this warp's O to the common row maximum and park it in the
        // scratch slot as fp32 [8 rows][128 dims]; the dim is XOR-swizzled
        // within its 16-group by (row >> 1, dim >> 5) so that both the
        // fragment-order stores and the dim-order loads are conflict-free.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = 2 * c + h;
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < NW; ++w) M = fmaxf(M, ms[w * 8 * NT + nt * 8 + row]);
          const float sc = (m_run[nt][h] == -INFINITY) ? 0.f : ex2(m_run[nt][h] - M);
          const int sw = (((g >> 1) & 3) | (c << 2));
#pragma unroll
          for (int mi = 0; mi < 8; ++mi) {
            const int d0 = 16 * g + mi, d1 = 16 * g + 8 + mi;
            stsf(myfree + (row * D + (d0 ^ sw)) * 4, o[nt][mi][h] * sc);
            stsf(myfree + (row * D + (d1 ^ sw)) * 4, o[nt][mi][2 + h] * sc);
          }
        }
        named_barrier(1, THREADS);
        {
          const int tid = threadIdx.x;   // = dim
          uint32_t fs[NW];
#pragma unroll
          for (int w = 0; w < NW; ++w) fs[w] = fslot[w];
          for (int r = 0; r < 8 && nt * 8 + r < p.qg; ++r) {
            const int row = nt * 8 + r;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NW; ++w) M = fmaxf(M, ms[w * 8 * NT + row]);
            float lsum = 0.f, acc = 0.f;
            const int pd = tid ^ (((tid >> 5) & 3) | ((r >> 1) << 2));
#pragma unroll
            for (int w = 0; w < NW; ++w) {
              const float mw = ms[w * 8 * NT + row];
              const float wt = (mw == -INFINITY) ? 0.f : ex2(mw - M);
              lsum += wt * ls[w * 8 * NT + row];
              acc += ldsf(fs[w] + (r * D + pd) * 4);
            }
            p.part_o[(row0 + row) * D + tid] = lsum > 0.f ? acc / lsum * vscale : 0.f;
            if (tid == 0) {
              p.part_m[row0 + row] = M == -INFINITY ? -INFINITY : M * kLn2;
              p.part_l[row0 + row] = lsum;
            }
          }
        }
        named_barrier(1, THREADS);
      }
      cur_item = -1;
    }

    if (kind == EV_NONE) break;
    issue(e + DEPTH - 1);
    cp_async_wait<DEPTH - 1>();
    __syncwarp();
    const uint32_t slot = ring + (e % DEPTH) * SLOT_BYTES;

    if (kind == EV_ITEM) {
      cur_item = ea;
      const bool work = (ea % P) * TG < eb;
      // ---- query fragments: q row r = 8*nt + g, dims [32c, 32c+32), scaled
      // by a power of two (largest element in [2^14, 2^15)) and rounded to f16
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int r = nt * 8 + g;
        float x[32];
        if (work && r < p.qg) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 w4 = lds128(slot + r * 256 + 64 * c + 16 * j);
            const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              x[8 * j + 2 * k] = __uint_as_float(ws[k] << 16);
              x[8 * j + 2 * k + 1] = __uint_as_float(ws[k] & 0xffff0000u);
            }
          }
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) x[k] = 0.f;
        }
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(x[k]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        int a = 0;     // 2^a with amax * 2^a in [2^14, 2^15)
        if (amax > 0.f) {
          int ex;
          frexpf(amax, &ex);
          a = max(-126, min(127, 15 - ex));
        }
        const float up = __uint_as_float(uint32_t(127 + a) << 23);
        const float down = 1.0f / up;   // exact power of two
#pragma unroll
        for (int k = 0; k < 16; ++k) qf[nt][k] = f32x2_to_f16x2(x[2 * k] * up, x[2 * k + 1] * up);
        const float mine = down * base_scale;   // logit multiplier of row r
        rowc[nt][0] = __shfl_sync(0xffffffffu, mine, (2 * c) * 4);
        rowc[nt][1] = __shfl_sync(0xffffffffu, mine, (2 * c + 1) * 4);
        m_run[nt][0] = m_run[nt][1] = -INFINITY;
        l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
        for (int mi = 0; mi < 8; ++mi)
#pragma unroll
          for (int k = 0; k < 4; ++k) o[nt][mi][k] = 0.f;
      }
      __syncwarp();
      continue;   // (the __syncwarp above ends this iteration's reads of the slot)
    }

    // ---- EV_SLICE: 16 tokens [16*ea, 16*ea + 16) of the current item
    const int t0 = ea * SLICE;
    const int L = eb;
    const bool partial = t0 + SLICE > L;
    // K rows g and g+8, chunks 2c and 2c+1 (chunk j of row r is stored at j ^ (r & 7))
    const uint4 ka0 = lds128(slot + g * D + (((2 * c) ^ g) << 4));
    const uint4 ka1 = lds128(slot + g * D + (((2 * c + 1) ^ g) << 4));
    const uint4 kb0 = lds128(slot + (g + 8) * D + (((2 * c) ^ g) << 4));
    const uint4 kb1 = lds128(slot + (g + 8) * D + (((2 * c + 1) ^ g) << 4));
    // V rows 2c, 2c+1, 2c+8, 2c+9, chunk g
    uint4 v0 = lds128(slot + 2048 + (2 * c) * D + ((g ^ (2 * c)) << 4));
    uint4 v1 = lds128(slot + 2048 + (2 * c + 1) * D + ((g ^ (2 * c + 1)) << 4));
    uint4 v8 = lds128(slot + 2048 + (2 * c + 8) * D + ((g ^ (2 * c)) << 4));
    uint4 v9 = lds128(slot + 2048 + (2 * c + 9) * D + ((g ^ (2 * c + 1)) << 4));
    const uint32_t kr0[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
    const uint32_t kr8[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
    if (partial) {
      // V bytes past the end may be NaN codes: zero them (0 * NaN = NaN)
      const uint4 z = make_uint4(0, 0, 0, 0);
      if (t0 + 2 * c >= L) v0 = z;
      if (t0 + 2 * c + 1 >= L) v1 = z;
      if (t0 + 2 * c + 8 >= L) v8 = z;
      if (t0 + 2 * c + 9 >= L) v9 = z;
    }
    // V^T A fragments (f16): dim 16g+dd, token pairs (2c,2c+1) -> [dd][0], (2c+8,2c+9) -> [dd][1]
    uint32_t aT[16][2];
    {
      const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w};
      const uint32_t w1[4] = {v1.x, v1.y, v1.z, v1.w};
      const uint32_t w8[4] = {v8.x, v8.y, v8.z, v8.w};
      const uint32_t w9[4] = {v9.x, v9.y, v9.z, v9.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t lo01 = prmt(w0[j], w1[j], 0x5140), hi01 = prmt(w0[j], w1[j], 0x7362);
        const uint32_t lo89 = prmt(w8[j], w9[j], 0x5140), hi89 = prmt(w8[j], w9[j], 0x7362);
        aT[4 * j + 0][0] = e4m3x2_lo_to_f16x2(lo01);
        aT[4 * j + 1][0] = e4m3x2_hi_to_f16x2(lo01);
        aT[4 * j + 2][0] = e4m3x2_lo_to_f16x2(hi01);
        aT[4 * j + 3][0] = e4m3x2_hi_to_f16x2(hi01);
        aT[4 * j + 0][1] = e4m3x2_lo_to_f16x2(lo89);
        aT[4 * j + 1][1] = e4m3x2_hi_to_f16x2(lo89);
        aT[4 * j + 2][1] = e4m3x2_lo_to_f16x2(hi89);
        aT[4 * j + 3][1] = e4m3x2_hi_to_f16x2(hi89);
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      // S^T (16 tokens x 8 rows) = K q^T; k-step ks covers dims 32c+4ks+{0,1} | {2,3},
      // i.e. K word ks of rows g and g+8 (two chains)
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < 8; ks += 2) {
        mma_f16_16816(sa, e4m3x2_lo_to_f16x2(kr0[ks]), e4m3x2_lo_to_f16x2(kr8[ks]), e4m3x2_hi_to_f16x2(kr0[ks]),
                      e4m3x2_hi_to_f16x2(kr8[ks]), qf[nt][2 * ks], qf[nt][2 * ks + 1]);
        mma_f16_16816(sb, e4m3x2_lo_to_f16x2(kr0[ks + 1]), e4m3x2_lo_to_f16x2(kr8[ks + 1]),
                      e4m3x2_hi_to_f16x2(kr0[ks + 1]), e4m3x2_hi_to_f16x2(kr8[ks + 1]), qf[nt][2 * ks + 2],
                      qf[nt][2 * ks + 3]);
      }
      // logits (log2 units): token t0+g -> x0, x1; t0+g+8 -> x2, x3
      float x0 = (sa[0] + sb[0]) * rowc[nt][0];
      float x1 = (sa[1] + sb[1]) * rowc[nt][1];
      float x2 = (sa[2] + sb[2]) * rowc[nt][0];
      float x3 = (sa[3] + sb[3]) * rowc[nt][1];
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
      const float mn0 = fmaxf(m_run[nt][0], mx0), mn1 = fmaxf(m_run[nt][1], mx1);
      if (__any_sync(0xffffffffu, (mn0 > m_run[nt][0]) || (mn1 > m_run[nt][1]))) {
        const float a0 = ex2(m_run[nt][0] - mn0), a1 = ex2(m_run[nt][1] - mn1);
        l_run[nt][0] *= a0;
        l_run[nt][1] *= a1;
#pragma unroll
        for (int mi = 0; mi < 8; ++mi) {
          o[nt][mi][0] *= a0; o[nt][mi][1] *= a1;
          o[nt][mi][2] *= a0; o[nt][mi][3] *= a1;
        }
        m_run[nt][0] = mn0;
        m_run[nt][1] = mn1;
      }
      const float p0 = ex2(x0 - mn0), p1 = ex2(x1 - mn1);
      const float p2 = ex2(x2 - mn0), p3 = ex2(x3 - mn1);
      const uint32_t P01 = f32x2_to_f16x2(p0, p1);
      const uint32_t P23 = f32x2_to_f16x2(p2, p3);
      // the sum uses the same f16-rounded probabilities the PV product sees
      l_run[nt][0] += f16_lo_to_f32(P01) + f16_lo_to_f32(P23);
      l_run[nt][1] += f16_hi_to_f32(P01) + f16_hi_to_f32(P23);
      const uint32_t b0 = movmatrix_trans(P01);   // tokens 2c, 2c+1 of row g
      const uint32_t b1 = movmatrix_trans(P23);   // tokens 2c+8, 2c+9 of row g
      // O^T (dims x 8 rows) += V^T (dims x 16 tokens) P^T; m-tile mi holds
      // dims 16g+mi (row g) and 16g+8+mi (row g+8)
#pragma unroll
      for (int mi = 0; mi < 8; ++mi)
        mma_f16_16816(o[nt][mi], aT[mi][0], aT[mi + 8][0], aT[mi][1], aT[mi + 8][1], b0, b1);
    }
    __syncwarp();
  }
  cp_async_wait<0>();
}

// Flash-combine of the partitions ([PA] reduce kernel): one CTA per query
// row (seq, kv_head, r), see combine_row.
template <typename OutT>
__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_m,
               const float* __restrict__ part_l, OutT* __restrict__ out, int num_kv_heads, int qg,
               int num_partitions, long long out_stride_seq, long long out_stride_head) {
  extern __shared__ __align__(16) float sw[];
  __shared__ __align__(16) float vec[fp8::D];
  pdl_wait_primary();
  const int row = blockIdx.x;                 // ((seq * Hk) + kvh) * qg + r
  const int r = row % qg;
  const int sk = row / qg;                    // seq * Hk + kvh
  const int seq = sk / num_kv_heads, kvh = sk % num_kv_heads;
  combine_row<fp8::D>(part_o, part_m, part_l, (long long)sk * num_partitions * qg + r, qg, num_partitions, sw, vec);
  if (threadIdx.x < fp8::D / 4) {
    const int t = threadIdx.x;
    OutT* dst = out + seq * out_stride_seq + (long long)(kvh * qg + r) * out_stride_head + 4 * t;
    store4(dst, vec[4 * t], vec[4 * t + 1], vec[4 * t + 2], vec[4 * t + 3]);
  }
}

// ------------------------------------------------------------------ host side
cudaError_t launch_fp8_partition(const Fp8Launch& a, cudaStream_t stream) {
  Fp8Params p;
  p.q = static_cast<const uint16_t*>(a.q);
  p.kv = a.kv;
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
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
  p.softmax_scale = a.softmax_scale;
  const long long items = (long long)a.num_seqs * a.num_kv_heads * a.num_partitions;
  if (items <= 0) return cudaSuccess;
  if (a.qg <= 8) {
    const int smem = fp8::Smem<1>::total;
    const int grid = (int)std::min<long long>(items, (long long)fp8::ctas_per_sm<1>() * a.num_sms);
    cudaFuncSetAttribute(pa_fp8_partition_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    pa_fp8_partition_kernel<1><<<grid, fp8::THREADS, smem, stream>>>(p);
  } else {
    const int smem = fp8::Smem<2>::total;
    const int grid = (int)std::min<long long>(items, (long long)fp8::ctas_per_sm<2>() * a.num_sms);
    cudaFuncSetAttribute(pa_fp8_partition_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    pa_fp8_partition_kernel<2><<<grid, fp8::THREADS, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

template <typename OutT>
static cudaError_t launch_combine_t(const CombineLaunch& a, OutT* out, cudaStream_t stream) {
  const int grid = a.num_seqs * a.num_kv_heads * a.qg;
  const size_t smem = combine_smem_bytes(a.num_partitions);
  if (smem > 40 * 1024)
    cudaFuncSetAttribute(combine_kernel<OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
  return cudaLaunchKernelEx(&cfg, combine_kernel<OutT>, a.part_o, a.part_m, a.part_l, out, a.num_kv_heads,
                            a.qg, a.num_partitions, a.out_stride_seq, a.out_stride_head);
}

cudaError_t launch_combine(const CombineLaunch& a, cudaStream_t stream) {
  if (a.num_seqs * a.num_kv_heads * a.qg <= 0) return cudaSuccess;
  cudaError_t e = a.out_bf16 ? launch_combine_t(a, static_cast<__nv_bfloat16*>(a.out), stream)
                             : launch_combine_t(a, static_cast<float*>(a.out), stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qpa
