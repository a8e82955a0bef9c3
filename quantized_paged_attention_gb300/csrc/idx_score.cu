// NVFP4 paged index scorer: per (index head, query row, block) the maximum
// of the causally visible dot products q . k_t over the block's 128 tokens.
//
// What it computes follows the vLLM nvfp4_index_decode kernel page (PR 59747):
//  * a page of 9216 bytes holds 128 tokens: bytes 0..8191 are the e2m1 codes,
//    64 per token (dim 2i in the low nibble of byte i), bytes 8192..9215 the
//    e4m3 scales, 8 per token, one per 16 dims (load_tile: codes at 64 t,
//    scales after PAGE_CODES);
//  * row qoff of request r sees tokens t <= L - QL + qoff (score_cgs limits);
//  * the score of a block is the max of its column over the page (frag_max);
//    blocks past the end of the request are written as -inf. A flag keeps
//    the dots before that max instead: one column per token, -inf where the
//    token is not visible.
//
// GB300 design:
//  * persistent CTAs of 4 warps; the (request, block) pages are split into
//    equal contiguous ranges, one per warp (found by a scan of seq_lens in
//    the kernel), so consecutive pages of a warp mostly share a request and
//    its query fragments, and the load is balanced to one page;
//  * each warp streams half pages (4 KB of codes + 512 B of scales) through a
//    private 4-slot cp.async ring (L2 evict-first); the block table is read
//    one page ahead;
//  * K is dequantised exactly to f16 (cvt e2m1x2, times the group scale with
//    hmul2: e2m1 x e4m3 has at most 6 significant bits) and multiplied with
//    the query rows (e4m3 -> f16, exact) on f16 mma.sync, m16n8k16 tiles of
//    16 tokens x 8 query rows; masking is by selection, the block max is a
//    register max plus a 3-step shuffle reduction.
#include <type_traits>

#include "common.cuh"
#include "qpa_internal.h"

namespace qpa {

namespace idx {
constexpr int BLK = 128;          // tokens per page
constexpr int PAGE_CODES = 8192;
constexpr int NW = 4;
constexpr int THREADS = NW * 32;
constexpr int DEPTH = 4;
constexpr int HALF_CODES = 4096;  // 64 tokens x 64 B
constexpr int HALF_SCALES = 512;  // 64 tokens x 8 B
constexpr int SLOT_BYTES = HALF_CODES + HALF_SCALES;   // 4608 (query rows need <= 2048)
constexpr int SMEM = NW * DEPTH * SLOT_BYTES;
constexpr int CTAS_PER_SM = 3;
}  // namespace idx

enum : int { IEV_NONE = 0, IEV_ITEM = 1, IEV_HALF = 2 };

template <int NT, bool PER_TOKEN>
__global__ void __launch_bounds__(idx::THREADS, idx::CTAS_PER_SM)
idx_score_kernel(const IdxParams p) {
  using namespace idx;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int R = p.num_reqs, QL = p.query_len, H = p.num_heads, S = p.num_cols;
  const int rows = QL * H;
  const uint64_t pol = policy_evict_first();
  const uint32_t ring = smem_u32(smem) + warp * DEPTH * SLOT_BYTES;
  const int col_blocks = PER_TOKEN ? (S + BLK - 1) / BLK : S;   // blocks that own a column
  auto nblocks = [&](int L) { return min((max(L, 0) + BLK - 1) / BLK, col_blocks); };
  const long long GW = (long long)gridDim.x * NW;
  const long long gw = (long long)blockIdx.x * NW + warp;

  // ---- columns past each request's last block (and every column when L <= 0)
  // are -inf: units (request, row, 1024-column chunk) spread over all warps,
  // a warp's lanes on consecutive columns
  {
    constexpr int CH = 1024;
    const int chunks = (S + CH - 1) / CH;
    const long long fill_units = (long long)R * rows * chunks;
    for (long long u = gw; u < fill_units; u += GW) {
      const int ch = (int)(u % chunks);
      const long long rn = u / chunks;
      const int n = (int)(rn % rows), r = (int)(rn / rows);
      const int nb = nblocks(__ldg(p.seq_lens + r));
      const int col0 = max(min(PER_TOKEN ? nb * BLK : nb, S), ch * CH);
      const int col1 = min(S, (ch + 1) * CH);
      float* row = p.scores + (n % H) * p.s_stride_head + (long long)(r * QL + n / H) * p.s_stride_row;
      for (int col = col0 + lane; col < col1; col += 32) row[col] = -INFINITY;
    }
  }

  // ---- this warp's page range: units u in [u0, u1) over (r, b), b < nblocks(L_r)
  long long U = 0;
  for (int r0 = 0; r0 < R; r0 += 32) {
    const int r = r0 + lane;
    int nb = r < R ? nblocks(__ldg(p.seq_lens + r)) : 0;
#pragma unroll
    for (int sh = 16; sh; sh >>= 1) nb += __shfl_xor_sync(0xffffffffu, nb, sh);
    U += nb;
  }
  const long long u0 = U * gw / GW, u1 = U * (gw + 1) / GW;
  // locate u0: request r_cur with prefix(r_cur) <= u0 < prefix(r_cur + 1)
  int r_cur = 0, b_cur = 0, L_cur = 0;
  {
    long long base = 0;
    bool found = false;
    for (int r0 = 0; r0 < R && !found; r0 += 32) {
      const int r = r0 + lane;
      const int L = r < R ? __ldg(p.seq_lens + r) : 0;
      const int nb = r < R ? nblocks(L) : 0;
      int incl = nb;   // inclusive scan over the 32 lanes
#pragma unroll
      for (int sh = 1; sh < 32; sh <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, sh);
        if (lane >= sh) incl += t;
      }
      const long long lo = base + incl - nb, hi = base + incl;
      const unsigned hit = __ballot_sync(0xffffffffu, r < R && u0 >= lo && u0 < hi);
      if (hit) {
        const int src = __ffs(hit) - 1;
        r_cur = r0 + src;
        b_cur = (int)(u0 - __shfl_sync(0xffffffffu, lo, src));
        L_cur = __shfl_sync(0xffffffffu, L, src);
        found = true;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
  }

  // ---------------------------------------------------------------- issue side
  // Events: an item event when the request changes (copies its query rows),
  // then two half-page events per page. Lane (e % DEPTH) keeps event e's record.
  long long iu = u0;
  int ir = r_cur, ib = b_cur, iL = L_cur, ihalf = 0, last_req = -1;
  int32_t iphys = 0;
  bool phys_ready = false;
  int rec_kind = 0, rec_r = 0, rec_bh = 0, rec_L = 0;

  auto load_phys = [&](int r, int b) -> int32_t {
    return __ldg(p.block_table + (long long)r * p.max_blocks + b);
  };
  auto advance_page = [&]() {   // to the next unit of the warp's range
    ++iu;
    if (++ib >= nblocks(iL)) {
      do {
        ++ir;
        iL = ir < R ? __ldg(p.seq_lens + ir) : 0;
      } while (ir < R && nblocks(iL) == 0);
      ib = 0;
    }
  };

  auto issue = [&](int e) {
    const uint32_t slot = ring + (e % DEPTH) * SLOT_BYTES;
    int kind = IEV_NONE, a = 0, bh = 0, lv = 0;
    if (iu < u1) {
      if (ir != last_req) {
        // query rows n = qoff * H + h of request ir: rows x 128 B
        for (int i = lane; i < rows * 8; i += 32) {
          const int n = i >> 3, ch = i & 7;
          const uint8_t* src = p.q + (long long)(ir * QL + n / H) * p.q_stride_tok + (long long)(n % H) * p.q_stride_head;
          cp_async16(slot + n * 128 + ch * 16, src + ch * 16, pol);
        }
        last_req = ir;
        kind = IEV_ITEM; a = ir; lv = iL;
      } else {
        if (!phys_ready) { iphys = load_phys(ir, ib); phys_ready = true; }
        int phys = iphys;
        if (phys < 0 || phys >= p.num_blocks) {
          if (lane == 0) atomicExch(&g_kernel_error, KERR_BAD_BLOCK);
          phys = 0;
        }
        const uint8_t* pg = p.pages + (long long)phys * p.page_stride;
        // 4096 B of codes + 512 B of scales of tokens [64 half, 64 half + 64)
        cp_async_halfpage(slot + 16 * lane, slot + HALF_CODES + 16 * lane, pg + ihalf * HALF_CODES + 16 * lane,
                          pg + PAGE_CODES + ihalf * HALF_SCALES + 16 * lane, pol);
        kind = IEV_HALF; a = ir; bh = (ib << 1) | ihalf; lv = iL;
        if (ihalf == 1) {
          advance_page();
          // table entry of the next page, in flight while this one streams
          phys_ready = false;
          if (iu < u1 && ir == last_req) { iphys = load_phys(ir, ib); phys_ready = true; }
        }
        ihalf ^= 1;
      }
    }
    cp_async_commit();
    if (lane == e % DEPTH) { rec_kind = kind; rec_r = a; rec_bh = bh; rec_L = lv; }
  };

  // ---------------------------------------------------------------- consume side
  const int g = lane >> 2;
  const int c = lane & 3;
  // this lane's accumulator rows n = 8 nt + 2c + hh: query offset n / H and
  // the score row's offset without the request's (divisions once, not per tile)
  int qo[NT][2];
  long long ro[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int n = nt * 8 + 2 * c + hh;
      qo[nt][hh] = n / H;
      ro[nt][hh] = (long long)(n % H) * p.s_stride_head + (long long)qo[nt][hh] * p.s_stride_row;
    }
  const long long req_stride = (long long)QL * p.s_stride_row;
  uint32_t qf[NT][16];     // query row 8 nt + g, dims [32c, 32c+32), f16x2
  float mx[NT][2];         // running block max of rows 8nt+2c, 8nt+2c+1

#pragma unroll 1
  for (int e = 0; e < DEPTH - 1; ++e) issue(e);

#pragma unroll 1
  for (int e = 0;; ++e) {
    const int kind = __shfl_sync(0xffffffffu, rec_kind, e % DEPTH);
    const int er = __shfl_sync(0xffffffffu, rec_r, e % DEPTH);
    const int ebh = __shfl_sync(0xffffffffu, rec_bh, e % DEPTH);
    const int eL = __shfl_sync(0xffffffffu, rec_L, e % DEPTH);
    if (kind == IEV_NONE) break;
    issue(e + DEPTH - 1);
    cp_async_wait<DEPTH - 1>();
    __syncwarp();
    const uint32_t slot = ring + (e % DEPTH) * SLOT_BYTES;

    if (kind == IEV_ITEM) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int n = nt * 8 + g;
        if (n < rows) {
          const uint4 w0 = lds128(slot + n * 128 + 32 * c), w1 = lds128(slot + n * 128 + 32 * c + 16);
          const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            qf[nt][2 * j] = e4m3x2_lo_to_f16x2(ws[j]);
            qf[nt][2 * j + 1] = e4m3x2_hi_to_f16x2(ws[j]);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) qf[nt][j] = 0u;
        }
      }
      __syncwarp();
      continue;
    }

    // ---- IEV_HALF: tokens [64 half, 64 half + 64) of block b of request er
    const int b = ebh >> 1, half = ebh & 1;
    if (half == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mx[nt][0] = mx[nt][1] = -INFINITY;
    }
    const int tok_base = b * BLK + 64 * half;
    const int last0 = eL - QL;    // row qoff sees tokens <= last0 + qoff
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int ra = 16 * m + g, rb = ra + 8;
      const uint4 ka = lds128(slot + ra * 64 + 16 * c), kb = lds128(slot + rb * 64 + 16 * c);
      const uint32_t sa = e4m3x2_lo_to_f16x2(lds32(slot + HALF_CODES + ra * 8 + 4 * (c >> 1)) >> (16 * (c & 1)));
      const uint32_t sb = e4m3x2_lo_to_f16x2(lds32(slot + HALF_CODES + rb * 8 + 4 * (c >> 1)) >> (16 * (c & 1)));
      const uint32_t sa0 = prmt(sa, sa, 0x1010), sa1 = prmt(sa, sa, 0x3232);
      const uint32_t sb0 = prmt(sb, sb, 0x1010), sb1 = prmt(sb, sb, 0x3232);
      const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w}, wb[4] = {kb.x, kb.y, kb.z, kb.w};
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t gsa = j < 2 ? sa0 : sa1, gsb = j < 2 ? sb0 : sb1;
        const uint32_t a0 = hmul2(e2m1x2_to_f16x2<0>(wa[j]), gsa), a2 = hmul2(e2m1x2_to_f16x2<1>(wa[j]), gsa);
        const uint32_t a4 = hmul2(e2m1x2_to_f16x2<2>(wa[j]), gsa), a6 = hmul2(e2m1x2_to_f16x2<3>(wa[j]), gsa);
        const uint32_t b0 = hmul2(e2m1x2_to_f16x2<0>(wb[j]), gsb), b2 = hmul2(e2m1x2_to_f16x2<1>(wb[j]), gsb);
        const uint32_t b4 = hmul2(e2m1x2_to_f16x2<2>(wb[j]), gsb), b6 = hmul2(e2m1x2_to_f16x2<3>(wb[j]), gsb);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          // k-step 2j: dims 32c+8j+{0,1} | {2,3}; k-step 2j+1: dims +{4,5} | {6,7}
          mma_f16_16816(acc[nt], a0, b0, a2, b2, qf[nt][4 * j], qf[nt][4 * j + 1]);
          mma_f16_16816(acc[nt], a4, b4, a6, b6, qf[nt][4 * j + 2], qf[nt][4 * j + 3]);
        }
      }
      const int ta = tok_base + 16 * m + g, tb = ta + 8;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int n = nt * 8 + 2 * c + hh;
          const int lim = last0 + qo[nt][hh];
          const float va = ta <= lim ? acc[nt][hh] : -INFINITY;
          const float vb = tb <= lim ? acc[nt][2 + hh] : -INFINITY;
          if constexpr (PER_TOKEN) {
            // 8 lanes of equal c write 8 consecutive tokens of one row
            if (n < rows) {
              float* row = p.scores + er * req_stride + ro[nt][hh];
              if (ta < S) row[ta] = va;
              if (tb < S) row[tb] = vb;
            }
          } else {
            mx[nt][hh] = fmaxf(mx[nt][hh], fmaxf(va, vb));
          }
        }
      }
    }
    if (!PER_TOKEN && half == 1) {
      // block done: reduce over the 8 token lanes and store
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v = mx[nt][hh];
#pragma unroll
          for (int sh = 4; sh < 32; sh <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, sh));
          const int n = nt * 8 + 2 * c + hh;
          if (g == 0 && n < rows) p.scores[er * req_stride + ro[nt][hh] + b] = v;
        }
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
}

// ---------------------------------------------------------------------------
// Shared-page variant (QPA_IDX_SHARED_PAGES): the [IDX] launch loop's dedup.
// Requests form groups of 8; a work pair is (group, block position b). For a
// pair, lanes 0..7 hold the group's block ids at b, __match_any_sync groups
// equal ids, and each distinct page is loaded and dequantised once and scored
// for every request of the group that maps it. Pairs are dealt to CTAs
// round-robin (position-major), so every SM gets a mix of shared and unshared
// positions; the distinct pages of a CTA's pairs go to its warps in turn.
// A job is one distinct page and up to MC of the requests mapping it (a page
// that more requests map is several jobs): the page is loaded once per job
// and each 16-token tile dequantised once for the job's requests, whose query
// fragments and block maxima stay in registers. Per warp: two page slots, the
// next page streaming in while the current one is scored.
namespace idxd {
constexpr int RGS = 8;            // requests per group
constexpr int NW = 4;
constexpr int THREADS = NW * 32;
constexpr int PAGE = 9216;
constexpr int SLOTS = 2;
constexpr int WARP_BYTES = SLOTS * PAGE;
constexpr int SMEM = NW * WARP_BYTES;
constexpr int CTAS_PER_SM = 3;
}  // namespace idxd

template <int NT, bool PER_TOKEN>
__global__ void __launch_bounds__(idxd::THREADS, idxd::CTAS_PER_SM)
idx_score_shared_kernel(const IdxParams p) {
  using namespace idxd;
  // requests scored per job with their query fragments in registers: a
  // tile is dequantised once for up to MC of a page's requests
  constexpr int MC = NT == 1 ? 4 : 2;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int R = p.num_reqs, QL = p.query_len, H = p.num_heads, S = p.num_cols;
  const int rows = QL * H;
  const uint64_t pol = policy_evict_first();
  const uint32_t wbase = smem_u32(smem) + warp * WARP_BYTES;
  const int col_blocks = PER_TOKEN ? (S + idx::BLK - 1) / idx::BLK : S;
  auto nblocks = [&](int L) { return min((max(L, 0) + idx::BLK - 1) / idx::BLK, col_blocks); };
  const long long GW = (long long)gridDim.x * NW;
  const long long gw = (long long)blockIdx.x * NW + warp;

  // ---- columns past each request's last block are -inf (as the plain kernel)
  {
    constexpr int CH = 1024;
    const int chunks = (S + CH - 1) / CH;
    const long long fill_units = (long long)R * rows * chunks;
    for (long long u = gw; u < fill_units; u += GW) {
      const int ch = (int)(u % chunks);
      const long long rn = u / chunks;
      const int n = (int)(rn % rows), r = (int)(rn / rows);
      const int nb = nblocks(__ldg(p.seq_lens + r));
      const int col0 = max(min(PER_TOKEN ? nb * idx::BLK : nb, S), ch * CH);
      const int col1 = min(S, (ch + 1) * CH);
      float* row = p.scores + (n % H) * p.s_stride_head + (long long)(r * QL + n / H) * p.s_stride_row;
      for (int col = col0 + lane; col < col1; col += 32) row[col] = -INFINITY;
    }
  }

  // ---- this warp's jobs: distinct pages of the CTA's pairs, every NW-th one
  const int NG = (R + RGS - 1) / RGS;
  const long long NP = (long long)NG * min(p.max_blocks, col_blocks);
  long long v = blockIdx.x;          // the CTA's current pair
  int pc = 0;                        // the CTA's distinct pages so far
  unsigned pend = 0;                 // leaders of the current pair not yet dealt
  int32_t pbid = 0;                  // this lane's block id at the current pair (lanes < RGS)
  unsigned pmatch = 0;
  unsigned pleft = 0;                // requests of the current page not yet dealt
  // the next pair's length and table entry of this lane's request, loaded one
  // pair ahead (the entry is inside the table's row even when b is past L)
  int nL = 0;
  int32_t nbid = 0;
  auto prefetch_pair = [&](long long vv) {
    if (vv < NP && lane < RGS) {
      const int b = (int)(vv / NG), req = (int)(vv % NG) * RGS + lane;
      if (req < R) {
        nL = __ldg(p.seq_lens + req);
        nbid = __ldg(p.block_table + (long long)req * p.max_blocks + b);
      }
    }
  };
  prefetch_pair(v);
  struct Job { int b, grp, page; unsigned mappers; };
  // next job of this warp, or page < 0 when there is none
  auto next_job = [&]() -> Job {
    while (true) {
      while (pend == 0) {
        if (v >= NP) return Job{0, 0, -1, 0u};
        const int b = (int)(v / NG), grp = (int)(v % NG);
        const int req = grp * RGS + lane;
        const bool act = lane < RGS && req < R && b < nblocks(nL);
        int32_t bid = -2 - lane;     // inactive lanes: ids no page has
        if (act) {
          bid = nbid;
          if (bid < 0 || bid >= p.num_blocks) {
            atomicExch(&g_kernel_error, KERR_BAD_BLOCK);
            bid = 0;
          }
        }
        prefetch_pair(v + gridDim.x);
        pbid = bid;
        pmatch = __match_any_sync(0xffffffffu, bid);
        pend = __ballot_sync(0xffffffffu, act && lane == __ffs(pmatch) - 1);
        if (pend == 0) v += gridDim.x;
      }
      // the next chunk of at most MC of the current page's requests
      const int lead = __ffs(pend) - 1;
      if (pleft == 0) pleft = __shfl_sync(0xffffffffu, pmatch, lead);
      unsigned chunk = 0;
#pragma unroll
      for (int i = 0; i < MC; ++i)
        if (pleft) {
          chunk |= pleft & (0u - pleft);
          pleft &= pleft - 1;
        }
      if (pleft == 0) pend &= pend - 1;
      const int mine = (pc++ % NW) == warp;
      const Job j{(int)(v / NG), (int)(v % NG), __shfl_sync(0xffffffffu, pbid, lead), chunk};
      if (pend == 0) v += gridDim.x;
      if (mine) return j;
    }
  };
  auto load_page = [&](uint32_t slot, int page) {
    const uint8_t* pg = p.pages + (long long)page * p.page_stride;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      cp_async_halfpage(slot + h * idx::HALF_CODES + 16 * lane, slot + idx::PAGE_CODES + h * idx::HALF_SCALES + 16 * lane,
                        pg + h * idx::HALF_CODES + 16 * lane, pg + idx::PAGE_CODES + h * idx::HALF_SCALES + 16 * lane, pol);
  };

  const int g = lane >> 2;
  const int c = lane & 3;
  // this lane's accumulator rows n = 8 nt + 2c + hh: query offset n / H and
  // the score row's offset without the request's
  int qo[NT][2];
  long long ro[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int n = nt * 8 + 2 * c + hh;
      qo[nt][hh] = n / H;
      ro[nt][hh] = (long long)(n % H) * p.s_stride_head + (long long)qo[nt][hh] * p.s_stride_row;
    }
  const long long req_stride = (long long)QL * p.s_stride_row;
  // query fragments of the job's requests: row 8 nt + g, dims [32c, 32c+32), f16x2
  uint32_t qf[MC][NT][16];
  auto load_q = [&](int slot_i, int req) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int n = nt * 8 + g;
      uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0;
      if (n < rows) {
        const uint8_t* src = p.q + (long long)(req * QL + n / H) * p.q_stride_tok + (long long)(n % H) * p.q_stride_head + 32 * c;
        w0 = __ldg(reinterpret_cast<const uint4*>(src));
        w1 = __ldg(reinterpret_cast<const uint4*>(src + 16));
      }
      const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        qf[slot_i][nt][2 * j] = e4m3x2_lo_to_f16x2(ws[j]);
        qf[slot_i][nt][2 * j + 1] = e4m3x2_hi_to_f16x2(ws[j]);
      }
    }
  };

  Job cur = next_job();
  if (cur.page >= 0) load_page(wbase, cur.page);
  cp_async_commit();
  for (int jn = 0; cur.page >= 0; ++jn) {
    const Job nxt = next_job();
    const uint32_t slot = wbase + (jn & 1) * PAGE;
    if (nxt.page >= 0) load_page(wbase + ((jn + 1) & 1) * PAGE, nxt.page);
    cp_async_commit();
    const int b = cur.b;
    // the job's requests (lanes of the group, lowest first)
    int reqs[MC], last0[MC];
    int nreq = 0;
    {
      unsigned mm = cur.mappers;
#pragma unroll
      for (int i = 0; i < MC; ++i) {
        reqs[i] = mm ? cur.grp * RGS + __ffs(mm) - 1 : -1;
        if (mm) { mm &= mm - 1; ++nreq; }
      }
    }
#pragma unroll
    for (int i = 0; i < MC; ++i)
      if (i < nreq) {
        load_q(i, reqs[i]);
        last0[i] = __ldg(p.seq_lens + reqs[i]) - QL;    // row qoff sees tokens <= last0 + qoff
      }
    cp_async_wait<1>();
    __syncwarp();
    // the page's tiles for exactly K requests (no predicated-off MMAs)
    auto score = [&](auto kc) {
      constexpr int K = decltype(kc)::value;
      float mx[K][NT][2];
#pragma unroll
      for (int i = 0; i < K; ++i)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mx[i][nt][0] = mx[i][nt][1] = -INFINITY;
#pragma unroll (K == 1 ? 2 : 1)
      for (int mt = 0; mt < 8; ++mt) {           // 16-token tiles of the page
        const int half = mt >> 2, m = mt & 3;
        const uint32_t hs = slot + half * idx::HALF_CODES;
        const uint32_t ss = slot + idx::PAGE_CODES + half * idx::HALF_SCALES;
        const int ra = 16 * m + g, rb = ra + 8;
        const uint4 ka = lds128(hs + ra * 64 + 16 * c), kb = lds128(hs + rb * 64 + 16 * c);
        const uint32_t sa = e4m3x2_lo_to_f16x2(lds32(ss + ra * 8 + 4 * (c >> 1)) >> (16 * (c & 1)));
        const uint32_t sb = e4m3x2_lo_to_f16x2(lds32(ss + rb * 8 + 4 * (c >> 1)) >> (16 * (c & 1)));
        const uint32_t sa0 = prmt(sa, sa, 0x1010), sa1 = prmt(sa, sa, 0x3232);
        const uint32_t sb0 = prmt(sb, sb, 0x1010), sb1 = prmt(sb, sb, 0x3232);
        const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w}, wb[4] = {kb.x, kb.y, kb.z, kb.w};
        float acc[K][NT][4];
#pragma unroll
        for (int i = 0; i < K; ++i)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) acc[i][nt][0] = acc[i][nt][1] = acc[i][nt][2] = acc[i][nt][3] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t gsa = j < 2 ? sa0 : sa1, gsb = j < 2 ? sb0 : sb1;
          const uint32_t a0 = hmul2(e2m1x2_to_f16x2<0>(wa[j]), gsa), a2 = hmul2(e2m1x2_to_f16x2<1>(wa[j]), gsa);
          const uint32_t a4 = hmul2(e2m1x2_to_f16x2<2>(wa[j]), gsa), a6 = hmul2(e2m1x2_to_f16x2<3>(wa[j]), gsa);
          const uint32_t b0 = hmul2(e2m1x2_to_f16x2<0>(wb[j]), gsb), b2 = hmul2(e2m1x2_to_f16x2<1>(wb[j]), gsb);
          const uint32_t b4 = hmul2(e2m1x2_to_f16x2<2>(wb[j]), gsb), b6 = hmul2(e2m1x2_to_f16x2<3>(wb[j]), gsb);
#pragma unroll
          for (int i = 0; i < K; ++i)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              // k-step 2j: dims 32c+8j+{0,1} | {2,3}; k-step 2j+1: dims +{4,5} | {6,7}
              mma_f16_16816(acc[i][nt], a0, b0, a2, b2, qf[i][nt][4 * j], qf[i][nt][4 * j + 1]);
              mma_f16_16816(acc[i][nt], a4, b4, a6, b6, qf[i][nt][4 * j + 2], qf[i][nt][4 * j + 3]);
            }
        }
        const int ta = b * idx::BLK + 16 * mt + g, tb = ta + 8;
#pragma unroll
        for (int i = 0; i < K; ++i) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int lim = last0[i] + qo[nt][hh];
              const float va = ta <= lim ? acc[i][nt][hh] : -INFINITY;
              const float vb = tb <= lim ? acc[i][nt][2 + hh] : -INFINITY;
              if constexpr (PER_TOKEN) {
                if (nt * 8 + 2 * c + hh < rows) {
                  float* row = p.scores + reqs[i] * req_stride + ro[nt][hh];
                  if (ta < S) row[ta] = va;
                  if (tb < S) row[tb] = vb;
                }
              } else {
                mx[i][nt][hh] = fmaxf(mx[i][nt][hh], fmaxf(va, vb));
              }
            }
          }
        }
      }
      if constexpr (!PER_TOKEN) {
        // block maxima: reduce over the 8 token lanes, lanes g == 0 store rows 8 nt + 2c + hh
#pragma unroll
        for (int i = 0; i < K; ++i)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              float v = mx[i][nt][hh];
#pragma unroll
              for (int sh = 4; sh < 32; sh <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, sh));
              const int n = nt * 8 + 2 * c + hh;
              if (g == 0 && n < rows)
                p.scores[reqs[i] * req_stride + ro[nt][hh] + b] = v;
            }
      }
    };
    if (nreq == 1) score(std::integral_constant<int, 1>{});
    else if (nreq == 2) score(std::integral_constant<int, 2>{});
    else if constexpr (MC > 2) {
      if (nreq == 3) score(std::integral_constant<int, 3>{});
      else score(std::integral_constant<int, MC>{});
    }
    __syncwarp();
    cur = nxt;
  }
  cp_async_wait<0>();
}

cudaError_t launch_idx_score(const IdxLaunch& a, cudaStream_t stream) {
  IdxParams p;
  p.q = a.q;
  p.pages = a.pages;
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  p.scores = a.scores;
  p.page_stride = a.page_stride;
  p.q_stride_tok = a.q_stride_tok;
  p.q_stride_head = a.q_stride_head;
  p.s_stride_head = a.s_stride_head;
  p.s_stride_row = a.s_stride_row;
  p.num_reqs = a.num_reqs;
  p.query_len = a.query_len;
  p.num_heads = a.num_heads;
  p.max_blocks = a.max_blocks;
  p.num_cols = a.num_cols;
  p.num_blocks = a.num_blocks;
  p.per_token = a.per_token;
  if (a.num_reqs <= 0 || a.num_cols <= 0) return cudaSuccess;
  const int grid = idx::CTAS_PER_SM * a.num_sms;
  auto launch = [&](auto kernel) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, idx::SMEM);
    kernel<<<grid, idx::THREADS, idx::SMEM, stream>>>(p);
  };
  const bool two = a.query_len * a.num_heads > 8;
  if (a.shared_pages) {
    const int sgrid = idxd::CTAS_PER_SM * a.num_sms;
    auto launch_s = [&](auto kernel) {
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, idxd::SMEM);
      kernel<<<sgrid, idxd::THREADS, idxd::SMEM, stream>>>(p);
    };
    if (a.per_token) {
      if (two) launch_s(idx_score_shared_kernel<2, true>); else launch_s(idx_score_shared_kernel<1, true>);
    } else {
      if (two) launch_s(idx_score_shared_kernel<2, false>); else launch_s(idx_score_shared_kernel<1, false>);
    }
    return cudaGetLastError();
  }
  if (a.per_token) {
    if (two) launch(idx_score_kernel<2, true>); else launch(idx_score_kernel<1, true>);
  } else {
    if (two) launch(idx_score_kernel<2, false>); else launch(idx_score_kernel<1, false>);
  }
  return cudaGetLastError();
}

}  // namespace qpa
