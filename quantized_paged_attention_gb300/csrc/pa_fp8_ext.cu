// fp8 (e4m3fn) paged-attention decode of query_len new tokens per sequence,
// with per-tensor or per-token K/V scales: split-KV partition kernel and
// flash-combine kernel.
//
// What it computes follows the ROCm/FlyDSL PR #825 page (the "per_token_kv"
// quantisation mode and the MTP query_length 1..4 commits): every cached
// (token, KV head) may carry its own K and V scale, and a sequence decodes
// query_len new tokens at once, query position qoff of a length-L sequence
// attending to the tokens t <= L - query_len + qoff (causal inside the query
// block; a row with no visible token in a tile contributes exactly 0). The
// scale layout [num_blocks][num_kv_heads][block_size] (one float per cached
// token, indexed like the cache) is this library's reading; the page names
// the mode but not a layout.
//
// GB300 design: persistent CTAs of four warps; inside an item (sequence, KV
// head, partition) warp w owns the 16-token slices 4k+w of every tile group
// and runs its own 16-byte cp.async ring of slices (K and V chunks, and the
// slice's 16 K and 16 V scales in per-token mode), so there is no cross-warp
// handshake on the stream. QK and PV run on f16 mma.sync m16n8k16 with K and
// V converted exactly from e4m3 in registers; the query rows are the
// query_len x query_group rows of a KV head (up to 16, two 8-row MMA tiles),
// each scaled by a power of two and rounded to f16. Per token, the K scale
// multiplies the logit and the V scale the probability that enters the PV
// product (not the softmax sum). At the end of an item the four warps' states
// merge in a fixed order. The per-tensor, one-query-token path of the library
// is the tcgen05 kernel of pa_fp8.cu; this kernel serves the wider modes.
#include "common.cuh"
#include "qpa_internal.h"
#include "combine.cuh"

namespace qpa {

namespace fp8x {
constexpr int D = 128;          // head_dim
constexpr int TG = 256;         // tile-group tokens (partition granule)
constexpr int SLICE = 16;       // tokens per warp step (one mma M tile)
constexpr int NW = 4;           // warps per CTA
constexpr int THREADS = NW * 32;
constexpr int DEPTH = 4;        // ring slots per warp (DEPTH-1 copy events in flight)
constexpr int KV_BYTES = 4096;  // one slice: K 2 KB + V 2 KB
constexpr int SC_OFF = KV_BYTES;             // 16 K scales then 16 V scales (per-token mode)
constexpr int SLOT_BYTES = KV_BYTES + 128;   // (an item's query rows need <= 16 x 256 B)

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
}  // namespace fp8x

struct Fp8ExtParams {
  const uint16_t* q;          // bf16 bits
  const uint8_t* kv;          // [NB][2][Hk][bs][128]
  const int32_t* block_table;
  const int32_t* seq_lens;
  const float* k_scale;       // [1], or [NB][Hk][bs] per token
  const float* v_scale;
  float* part_o;              // [B][Hk][P][rows][D]
  float* part_m;              // [B][Hk][P][rows]
  float* part_l;              // [B][Hk][P][rows]
  long long q_stride_seq, q_stride_tok, q_stride_head;   // elements
  int num_seqs, num_kv_heads, qg, query_len, rows, block_size, log2_bs, num_blocks, max_blocks, num_partitions;
  float softmax_scale;
};

enum : int { XEV_NONE = 0, XEV_ITEM = 1, XEV_SLICE = 2 };

template <int NT, bool PT>
__global__ void __launch_bounds__(fp8x::THREADS, fp8x::ctas_per_sm<NT>())
pa_fp8x_partition_kernel(const Fp8ExtParams p) {
  using namespace fp8x;
  using S = Smem<NT>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Hk = p.num_kv_heads;
  const int num_items = p.num_seqs * Hk * p.num_partitions;
  const int P = p.num_partitions;
  const int bs = p.block_size;
  const int lbs = p.log2_bs;
  const int bpt = TG / bs;                        // table entries per tile group
  float* ms = reinterpret_cast<float*>(smem + S::mOff);
  float* ls = reinterpret_cast<float*>(smem + S::lOff);
  uint32_t* fslot = reinterpret_cast<uint32_t*>(smem + S::fOff);
  pdl_launch_dependents();   // the combine kernel waits for this grid before reading

  const uint64_t pol = policy_evict_first();
  const uint32_t ring = smem_u32(smem + S::ringOff) + warp * DEPTH * SLOT_BYTES;
  const size_t head_bytes = size_t(bs) * D;                     // one (block, K/V, head) chunk
  const size_t v_off = size_t(Hk) * head_bytes;                 // K chunk -> V chunk
  const size_t blk_bytes = 2 * v_off;                           // one block: K and V of all heads

  // ---------------------------------------------------------------- issue side
  // The warp walks its own event stream: per item of this CTA an item event
  // (the item's query rows) and then the item's slices owned by this warp.
  // Events are issued DEPTH-1 ahead of their use; lane (e % DEPTH) keeps
  // event e's record.
  int ik_item = blockIdx.x;
  int i_state = 0;                // 0: item event next, 1: slices next
  int i_tg = 0, i_kk = 0;
  int i_L = 0, i_Lnext = 0;
  int i_seq = 0, i_kvh = 0, i_part = 0;
  int32_t i_ent = 0, i_nent = 0;  // table entries of the current / next tile group (lane j: entry j)
  size_t kvh_off = 0;
  int rec_a = 0, rec_b = 0;        // event record: (payload << 2) | kind, length
  const int l3 = lane >> 3, j8 = lane & 7;
  const uint32_t doff0 = l3 * D + ((j8 ^ l3) << 4);
  const uint32_t doff1 = l3 * D + ((j8 ^ (l3 | 4)) << 4);
  const uint32_t l16 = lane * 16;

  auto load_len = [&](int item) -> int {
    if (item >= num_items) return 0;
    const int seq = item / (P * Hk);
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
    int kind = XEV_NONE, a = 0, b = 0;
    while (true) {
      if (ik_item >= num_items) break;
      if (i_state == 0) {
        i_part = ik_item % P;
        const int t = ik_item / P;
        i_kvh = t % Hk;
        i_seq = t / Hk;
        kvh_off = size_t(i_kvh) * head_bytes;
        if (i_part * TG < i_L) {
          // query rows r = qoff * qg + g of (seq, kv_head): rows x 256 B, 16 B per copy
          const uint16_t* qbase = p.q + i_seq * p.q_stride_seq + (long long)(i_kvh * p.qg) * p.q_stride_head;
          for (int idx = lane; idx < p.rows * 16; idx += 32) {
            const int row = idx >> 4, ch = idx & 15;
            const int qoff = row / p.qg, g = row - qoff * p.qg;
            cp_async16(slot + row * 256 + ch * 16,
                       qbase + qoff * p.q_stride_tok + (long long)g * p.q_stride_head + ch * 8, pol);
          }
          i_ent = load_entries(i_seq, i_part, i_L);
          if ((i_part + P) * TG < i_L) i_nent = load_entries(i_seq, i_part + P, i_L);
        }
        i_state = 1;
        i_tg = i_part;
        i_kk = 0;
        kind = XEV_ITEM; a = ik_item; b = i_L;
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
      const int tin = (s * SLICE) & (bs - 1);      // slice's first slot in the block
      const uint8_t* kb = p.kv + size_t(phys) * blk_bytes + kvh_off + size_t(tin) * D + l16;
      cp_async_chunk_pair(slot + doff0, slot + doff1, kb, kb + v_off, pol);
      if (PT && lane < 8) {
        // the slice's 16 K scales (lanes 0..3) and 16 V scales (lanes 4..7)
        const float* sc = (lane < 4 ? p.k_scale : p.v_scale) + (size_t(phys) * Hk + i_kvh) * bs + tin;
        cp_async16(slot + SC_OFF + 16 * lane, sc + 4 * (lane & 3), pol);
      }
      kind = XEV_SLICE; a = s; b = i_L;
      break;
    }
    cp_async_commit();
    if (lane == e % DEPTH) { rec_a = (a << 2) | kind; rec_b = b; }
  };

  // ---------------------------------------------------------------- consume side
  const int g = lane >> 2;      // fragment group id (row within 8)
  const int c = lane & 3;       // thread within group
  const float kscale = PT ? 1.f : __ldg(p.k_scale);
  const float vscale = PT ? 1.f : __ldg(p.v_scale);
  const float base_scale = kscale * p.softmax_scale * kLog2e;

  uint32_t qf[NT][16];   // query row 8nt+g, dims [32c, 32c+32), scaled, f16x2
  float rowc[NT][2];     // logit multiplier of this lane's rows 8nt+2c, 8nt+2c+1
  int lim[NT][2];        // those rows see the tokens t < lim
  float o[NT][8][4];
  float m_run[NT][2], l_run[NT][2];
  int cur_item = -1;
  int vis = 0;           // tokens t < vis are visible to every query row

#pragma unroll 1
  for (int e = 0; e < DEPTH - 1; ++e) issue(e);

#pragma unroll 1
  for (int e = 0;; ++e) {
    const int ra = __shfl_sync(0xffffffffu, rec_a, e % DEPTH);
    const int eb = __shfl_sync(0xffffffffu, rec_b, e % DEPTH);
    const int kind = ra & 3, ea = ra >> 2;

    if (kind != XEV_SLICE && cur_item >= 0) {
      // ---- end of the current item: merge the four warps' (m, l, O) in a
      // fixed order and write this partition's partials.
      const long long row0 = (long long)cur_item * p.rows;
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
        // within its 16-group by (row >> 1, dim >> 5) so that the fragment-order
        // stores and the dim-order loads are conflict-free
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
          for (int r = 0; r < 8 && nt * 8 + r < p.rows; ++r) {
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

    if (kind == XEV_NONE) break;
    issue(e + DEPTH - 1);
    cp_async_wait<DEPTH - 1>();
    __syncwarp();
    const uint32_t slot = ring + (e % DEPTH) * SLOT_BYTES;

    if (kind == XEV_ITEM) {
      cur_item = ea;
      const int L = eb;
      const bool work = (ea % P) * TG < L;
      vis = L - p.query_len + 1;
      // ---- query fragments: row r = 8*nt + g, dims [32c, 32c+32), scaled by
      // a power of two (largest element in [2^14, 2^15)) and rounded to f16
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int r = nt * 8 + g;
        float x[32];
        if (work && r < p.rows) {
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
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = nt * 8 + 2 * c + h;
          lim[nt][h] = row < p.rows ? vis + row / p.qg : vis;
        }
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

    // ---- XEV_SLICE: 16 tokens [16*ea, 16*ea + 16) of the current item
    const int t0 = ea * SLICE;
    const int L = eb;
    const bool masked = t0 + SLICE > vis;         // some token is invisible to some row
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
    // per-token scales of this lane's logit tokens g, g+8 and probability
    // tokens g, g+8 (slots past the end may hold NaN: masked below by selection)
    float ksg = 1.f, ksg8 = 1.f, vsg = 1.f, vsg8 = 1.f;
    if (PT) {
      ksg = ldsf(slot + SC_OFF + 4 * g);
      ksg8 = ldsf(slot + SC_OFF + 4 * (g + 8));
      vsg = ldsf(slot + SC_OFF + 64 + 4 * g);
      vsg8 = ldsf(slot + SC_OFF + 64 + 4 * (g + 8));
    }
    if (t0 + SLICE > L) {
      // V bytes and scales past the end may be NaN codes: zero them (0 * NaN = NaN)
      const uint4 z = make_uint4(0, 0, 0, 0);
      if (t0 + 2 * c >= L) v0 = z;
      if (t0 + 2 * c + 1 >= L) v1 = z;
      if (t0 + 2 * c + 8 >= L) v8 = z;
      if (t0 + 2 * c + 9 >= L) v9 = z;
      if (t0 + g >= L) vsg = 0.f;
      if (t0 + g + 8 >= L) vsg8 = 0.f;
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
      // logits (log2 units): token t0+g -> x0, x1; t0+g+8 -> x2, x3 (rows 2c, 2c+1)
      float x0 = (sa[0] + sb[0]) * rowc[nt][0] * ksg;
      float x1 = (sa[1] + sb[1]) * rowc[nt][1] * ksg;
      float x2 = (sa[2] + sb[2]) * rowc[nt][0] * ksg8;
      float x3 = (sa[3] + sb[3]) * rowc[nt][1] * ksg8;
      if (masked) {
        if (t0 + g >= lim[nt][0]) x0 = -INFINITY;
        if (t0 + g >= lim[nt][1]) x1 = -INFINITY;
        if (t0 + g + 8 >= lim[nt][0]) x2 = -INFINITY;
        if (t0 + g + 8 >= lim[nt][1]) x3 = -INFINITY;
      }
      float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
      for (int sh = 4; sh < 32; sh <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
      }
      const float mn0 = fmaxf(m_run[nt][0], mx0), mn1 = fmaxf(m_run[nt][1], mx1);
      if (__any_sync(0xffffffffu, (mn0 > m_run[nt][0]) || (mn1 > m_run[nt][1]))) {
        const float a0 = (m_run[nt][0] == -INFINITY) ? 0.f : ex2(m_run[nt][0] - mn0);
        const float a1 = (m_run[nt][1] == -INFINITY) ? 0.f : ex2(m_run[nt][1] - mn1);
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
      // (a row that has seen no visible token yet keeps m = -inf: its
      // probabilities are exactly 0, never exp2(-inf - (-inf)))
      const float p0 = (mn0 == -INFINITY) ? 0.f : ex2(x0 - mn0);
      const float p1 = (mn1 == -INFINITY) ? 0.f : ex2(x1 - mn1);
      const float p2 = (mn0 == -INFINITY) ? 0.f : ex2(x2 - mn0);
      const float p3 = (mn1 == -INFINITY) ? 0.f : ex2(x3 - mn1);
      uint32_t P01, P23;
      if (PT) {
        // the V scale enters the PV product, not the softmax sum
        l_run[nt][0] += p0 + p2;
        l_run[nt][1] += p1 + p3;
        P01 = f32x2_to_f16x2(p0 * vsg, p1 * vsg);
        P23 = f32x2_to_f16x2(p2 * vsg8, p3 * vsg8);
      } else {
        P01 = f32x2_to_f16x2(p0, p1);
        P23 = f32x2_to_f16x2(p2, p3);
        // the sum uses the same f16-rounded probabilities the PV product sees
        l_run[nt][0] += f16_lo_to_f32(P01) + f16_lo_to_f32(P23);
        l_run[nt][1] += f16_hi_to_f32(P01) + f16_hi_to_f32(P23);
      }
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

// Flash-combine of the partitions ([PA] reduce) of one query row (sequence,
// KV head, query position, group row), see combine_row.
template <typename OutT>
__global__ void __launch_bounds__(kCombineMaxThreads)
combine_ext_kernel(const float* __restrict__ part_o, const float* __restrict__ part_m,
                   const float* __restrict__ part_l, OutT* __restrict__ out, int num_kv_heads, int qg,
                   int query_len, int num_partitions, long long out_stride_seq, long long out_stride_tok,
                   long long out_stride_head) {
  extern __shared__ __align__(16) float sw[];
  __shared__ __align__(16) float vec[fp8x::D];
  pdl_wait_primary();
  const int rows = query_len * qg;
  const int row = blockIdx.x;                 // ((seq * Hk) + kvh) * rows + r
  const int r = row % rows;
  const int sk = row / rows;                  // seq * Hk + kvh
  const int seq = sk / num_kv_heads, kvh = sk % num_kv_heads;
  const int qoff = r / qg, gq = r % qg;
  combine_row<fp8x::D, kCombineKmax128>(part_o, part_m, part_l, (long long)sk * num_partitions * rows + r, rows,
                                        num_partitions, sw, vec);
  if (threadIdx.x < fp8x::D / 4) {
    const int t = threadIdx.x;
    OutT* dst = out + seq * out_stride_seq + qoff * out_stride_tok + (long long)(kvh * qg + gq) * out_stride_head + 4 * t;
    store4(dst, vec[4 * t], vec[4 * t + 1], vec[4 * t + 2], vec[4 * t + 3]);
  }
}

// ------------------------------------------------------------------ host side
cudaError_t launch_fp8x_partition_mma(const Fp8ExtLaunch& a, cudaStream_t stream) {
  Fp8ExtParams p;
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
  p.q_stride_tok = a.q_stride_tok;
  p.q_stride_head = a.q_stride_head;
  p.num_seqs = a.num_seqs;
  p.num_kv_heads = a.num_kv_heads;
  p.qg = a.qg;
  p.query_len = a.query_len;
  p.rows = a.query_len * a.qg;
  p.block_size = a.block_size;
  p.log2_bs = 0;
  while ((1 << p.log2_bs) < a.block_size) ++p.log2_bs;
  p.num_blocks = a.num_blocks;
  p.max_blocks = a.max_blocks;
  p.num_partitions = a.num_partitions;
  p.softmax_scale = a.softmax_scale;
  const long long items = (long long)a.num_seqs * a.num_kv_heads * a.num_partitions;
  if (items <= 0) return cudaSuccess;
  auto launch = [&](auto kern, int smem, int per_sm) {
    const int grid = (int)std::min<long long>(items, (long long)per_sm * a.num_sms);
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    kern<<<grid, fp8x::THREADS, smem, stream>>>(p);
  };
  if (p.rows <= 8) {
    if (a.per_token) launch(pa_fp8x_partition_kernel<1, true>, fp8x::Smem<1>::total, fp8x::ctas_per_sm<1>());
    else launch(pa_fp8x_partition_kernel<1, false>, fp8x::Smem<1>::total, fp8x::ctas_per_sm<1>());
  } else {
    if (a.per_token) launch(pa_fp8x_partition_kernel<2, true>, fp8x::Smem<2>::total, fp8x::ctas_per_sm<2>());
    else launch(pa_fp8x_partition_kernel<2, false>, fp8x::Smem<2>::total, fp8x::ctas_per_sm<2>());
  }
  return cudaGetLastError();
}

template <typename OutT>
static cudaError_t launch_fp8x_combine_t(const Fp8ExtCombineLaunch& a, OutT* out, cudaStream_t stream) {
  const int rows = a.query_len * a.qg;
  const int grid = a.num_seqs * a.num_kv_heads * rows;
  const int threads = combine_threads(fp8x::D, kCombineKmax128, a.num_partitions);
  const size_t smem = combine_smem_bytes(a.num_partitions, threads);
  if (smem > 40 * 1024)
    cudaFuncSetAttribute(combine_ext_kernel<OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
  return cudaLaunchKernelEx(&cfg, combine_ext_kernel<OutT>, a.part_o, a.part_m, a.part_l, out, a.num_kv_heads,
                            a.qg, a.query_len, a.num_partitions, a.out_stride_seq, a.out_stride_tok,
                            a.out_stride_head);
}

cudaError_t launch_fp8x_combine(const Fp8ExtCombineLaunch& a, cudaStream_t stream) {
  if (a.num_seqs * a.num_kv_heads * a.query_len * a.qg <= 0) return cudaSuccess;
  cudaError_t e = a.out_bf16 ? launch_fp8x_combine_t(a, static_cast<__nv_bfloat16*>(a.out), stream)
                             : launch_fp8x_combine_t(a, static_cast<float*>(a.out), stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qpa
