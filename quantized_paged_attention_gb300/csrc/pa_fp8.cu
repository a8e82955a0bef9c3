// fp8 (e4m3fn) paged-attention decode: split-KV partition kernel (head_dim
// 64 or 128, up to 16 query rows per work stream and 64 per KV head, a
// multi-token / per-token-scale variant) and flash-combine kernel.
//
// What it computes follows the ROCm/FlyDSL PR #825 page ("perf(pa tile):
// readable tile-programming PA decode kernel": per-tensor fp8 K/V, query
// length 1, GQA, cross-CTA split of a sequence and a parallel flash-combine
// reduce), with 256-token tile groups as the split granule (the
// ultraquant_decode_hd256 page, STEP F).
//
// GB300 design (not the pages' AMD design): one persistent CTA per SM with
// three warp roles around the 5th-generation tensor core.
//  * Work split: a KV head with more than 16 query rows is RB = rows / 16
//    (rounded up) virtual heads that read its pages and each own 16 rows;
//    the CTAs form groups of Hk * RB, one per virtual head; the groups cut
//    each head's tile groups (in sequence order) into equal contiguous
//    ranges, so the CTAs of a group read the same pages together and every
//    CTA gets the same number of tile groups in a few items. The part of a
//    sequence inside one range is an item; its softmax state is one of the
//    num_partitions slots of the (sequence, head) (slot = range index minus
//    that of the sequence's first tile group), unused slots are marked empty,
//    and the combine merges the slots. The page's own map (partition p owns
//    tile groups p, p+P, ...) gives many short items on ragged batches.
//  * 4 copy warps stream the item's 128-token tiles (K 16 KB + V 16 KB) into a
//    ring of shared-memory slots with per-lane 16-byte cp.async (a page chunk
//    of block_size 16 is only 2 KB, far too small per copy for one TMA issuing
//    thread), XOR-swizzled so that each slot is the 128-byte-swizzle canonical
//    layout the tensor core reads; tokens past the sequence length are
//    zero-filled. The copy warps also build the item's query operand.
//  * a QK warp and a PV warp issue tcgen05.mma kind::f8f6f4 straight on the
//    e4m3 bytes: S^T = K Q'^T (M = 128 tokens, N = 32 or 64) and
//    O^T = V^T P'^T (M = 128 dims, N = 32 or 64), accumulators in tensor
//    memory (two S buffers, four O buffers with 8 rows, two with 16).
//  * two groups of 4 softmax warps: thread t owns tensor-memory lane t, i.e.
//    token t of an S tile and dim t of an O tile. With up to 8 query rows the
//    groups take alternate tiles and merge per item; with 16 rows each group
//    owns 8 rows of every tile and takes the tiles two at a time (one maxima
//    exchange, one rescale and one O fold per 256 tokens; the second tile's
//    PV accumulates onto the first's O). They turn S into probabilities
//    (online softmax across the item's tiles), write P' for the next MMA, and
//    fold each O buffer into per-dim register accumulators with the softmax
//    rescale.
// Exactness: the query (bf16) and the probabilities (f16) enter the fp8 MMA
// as sums of e4m3 terms with power-of-two weights -- 3 terms for p (exact for
// its f16 value); 4 terms for q, and 2 with 16 rows: a row scaled to max |q|
// in [128, 256) is then exact in every element of magnitude >= 2^-6 (down to
// 2^-14 of the row maximum), the others within 2^-14, i.e. 2^-21 of the row
// maximum (the 4 terms move that bound 2^-8 lower) -- so the tensor core sees
// K and V unconverted and the products carry no fp8 rounding of q or p above
// those bounds.
// Every wait has a time limit; a timeout raises the error word and all roles
// leave through the common teardown.
#include "qpa.h"
#include "common.cuh"
#include "qpa_internal.h"
#include "combine.cuh"
#include "tc.cuh"

namespace qpa {

namespace fp8 {
constexpr int D = 128;          // head_dim
constexpr int TG = 256;         // tile-group tokens (partition granule)
constexpr int TILE = 128;       // tokens per MMA tile
constexpr int TILE_BYTES = 2 * TILE * D;   // K tile then V tile
constexpr int V_OFF = TILE * D;

// PK (head_dim 64, up to 8 query rows, one token per row): a ring slot holds a
// whole 256-token tile group, its first 128 tokens in bytes 0..63 of the
// 128-byte rows and the next 128 in bytes 64..127 ("halves" A and B); the MMA
// N doubles (Q' and P' carry each row once per half) so that one QK and one
// PV issue cover both halves and the softmax takes 256 tokens per pass.
template <int NT, bool EXT = false, bool PK = false>
struct Smem {
  static constexpr int NWG = 2;                    // softmax warp groups
  static constexpr int WARP_PROD0 = 4 * NWG;       // 4 copy warps
  static constexpr int WARP_MMA = WARP_PROD0 + 4;  // QK issuing warp, then the PV issuing warp
  static constexpr int THREADS = (WARP_MMA + 2) * 32;
  // ring slots (tiles, PK: tile groups): as many as shared memory holds, since
  // about two of them are always held by the MMAs and the softmax
  static constexpr int NS = (NT == 1 && !EXT && !PK) ? 6 : 5;
  static constexpr int R = 8 * NT;                 // query rows (padded)
  static constexpr int NQ = 32 * NT;               // 4 term slots x R rows
  static constexpr int NQS = PK ? 2 * NQ : NQ;     // MMA N: NQ per half
  static constexpr int QT = NT == 2 ? 2 : 4;       // e4m3 terms of the query (16 rows: 2)
  static constexpr int NQK = NT == 2 ? 8 * QT * NT : NQS;   // QK N: QT terms x R rows (per half)
  static constexpr int qBytes = NQK * D;           // Q' [NQK rows][128 dims] e4m3
  static constexpr int pBytes = TILE * NQS;        // P'^T [128 tokens][NQS] e4m3
  static constexpr int ringOff = 0;
  static constexpr int qOff = NS * TILE_BYTES;
  static constexpr int pOff = qOff + 2 * qBytes;
  static constexpr int stgOff = pOff + 4 * pBytes;         // [2][R][128] f32 second group's O (8 rows)
  static constexpr int cOff = stgOff + (NT == 1 ? 2 * R * D * 4 : 0);   // [2][R] logit multiplier per row
  static constexpr int redOff = cOff + 2 * R * 4;          // [2 S buffers][row blocks][4 warps][8] tile maxima
  static constexpr int lredOff = redOff + 2 * 4 * R * 4;   // [2][8 warps][8] row sums per warp
  static constexpr int msmOff = lredOff + 2 * 4 * NWG * R * 4;   // [2][2 groups][8] row maxima per group
  static constexpr int infoOff = msmOff + 2 * NWG * R * 4; // [2] {item, L, tiles, first tile group}, {row block, ..}
  static constexpr int pdOff = infoOff + 2 * 32;           // [4] per P' buffer: O buffer, accumulate, commit (16 rows)
  static constexpr int scOff = pdOff + 16;                 // EXT: [NS][K, V][128] f32 per-token scales
  static constexpr int barOff = (scOff + (EXT ? NS * 2 * TILE * 4 : 0) + 7) & ~7;
  static constexpr int NBAR = 2 * NS + 27;
  static constexpr int miscOff = barOff + NBAR * 8;        // tmem base, abort flag, QK total
  static constexpr int total = miscOff + 16 + 1024;        // + alignment slack
  static_assert(total <= 227 * 1024, "shared memory");
  static constexpr int TMEM_COLS = (NT == 1 && !PK) ? 256 : 512;   // S[2] (NQK columns) then O[4] (NQS)
};
}  // namespace fp8

struct Fp8Params {
  const uint16_t* q;          // bf16 bits
  const uint8_t* kv;          // [NB][2][Hk][bs][head_dim]
  const int32_t* block_table;
  const int32_t* seq_lens;
  const float* k_scale;
  const float* v_scale;
  float* part_o;              // [B][Hk][P][rows][head_dim], rows = query_len * QG
  float* part_m;              // [B][Hk][P][rows]
  float* part_l;              // [B][Hk][P][rows]
  long long q_stride_seq, q_stride_head;   // elements
  int num_seqs, num_kv_heads, qg, block_size, log2_bs, num_blocks, max_blocks, num_partitions;
  float softmax_scale;
  // multi-token variant: query_len new tokens per sequence (row qoff * qg + g,
  // causal inside the query block), K/V scales per tensor or per token
  // ([num_blocks][Hk][block_size] in k_scale / v_scale)
  long long q_stride_tok;
  int query_len, per_token;
  // query rows per KV head above 16: blocks of 16 rows run as separate
  // "virtual heads" (KV head vh / row_blocks, rows 16 (vh % row_blocks) ..)
  int row_blocks;
  int test_flags;   // QPA_TEST_WITHHOLD_ARRIVAL: copy warp 0 withholds its first tile's arrival
};

// HD: the cache's head_dim (64 or 128). Shared-memory rows stay 128 bytes
// (the 128-byte-swizzle layout); with HD = 64 their upper half is zeroed once
// and never written, so the QK steps over it are skipped and the PV rows of
// dims 64..127 come out zero.
// EXT: the multi-token / per-token variant (query_len, per_token of the
// parameters); rows = query_len * qg per item, a causal limit per row, and
// with per-token scales the copy warps bring each tile's K and V scales into
// shared memory next to the tile.
template <int NT, int HD, bool EXT>
__global__ void __launch_bounds__(fp8::Smem<NT>::THREADS, 1)
pa_fp8_partition_kernel(const Fp8Params p) {
  using namespace fp8;
  constexpr bool PK = HD == 64 && NT == 1 && !EXT;   // two 128-token halves per ring slot
  constexpr bool RS = NT == 2;                        // 16 rows: row split, two tiles per softmax pass
  using S = Smem<NT, EXT, PK>;
  constexpr int R = S::R, NQ = S::NQ, NQS = S::NQS, NQK = S::NQK, QT = S::QT, NWG = S::NWG;
  constexpr int PD = PK ? 2 * HD : HD;                // floats per partial O row
  constexpr int WARP_PROD0 = S::WARP_PROD0, WARP_MMA = S::WARP_MMA;
  constexpr uint32_t IDESC_QK = idesc_e4m3(128, NQK, false, false);
  constexpr uint32_t IDESC_PV = idesc_e4m3(128, NQS, true, true);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;     // swizzle atoms need 1024-byte alignment
  uint8_t* sm = smem_raw + (sbase - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S::barOff);
  constexpr int NS = S::NS;
  uint64_t* full = bars;              // [NS] tile copied (128 copy lanes)
  uint64_t* empty = full + NS;        // [NS] tile consumed (MMA commit)
  uint64_t* qfull = empty + NS;       // [2] Q' built (4 copy warps)
  uint64_t* qempty = qfull + 2;       // [2] Q' consumed (MMA commit + softmax warps)
  uint64_t* sfull = qempty + 2;       // [2] S tile ready (MMA commit)
  uint64_t* sfree = sfull + 2;        // [2] S tile read (4 softmax warps)
  uint64_t* pfull = sfree + 2;        // [4] P' buffer written (4 softmax warps)
  uint64_t* ofull = pfull + 4;        // [4] O buffer ready (PV commit)
  uint64_t* xbar = ofull + 4;         // [2 S buffers][2 row blocks] tile maxima exchanged (a group's 4 warps)
  uint64_t* merge = xbar + 4;         // [2][2] item states published (softmax warps)
  uint64_t* mfree = merge + 4;        // [2] item states read (the merging group's 4 warps)
  uint64_t* done = mfree + 2;         // [1] all MMAs finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S::miscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + S::miscOff + 4);
  volatile int* qk_total = reinterpret_cast<volatile int*>(sm + S::miscOff + 8);   // tiles, once all QKs are issued
  const uint32_t cbuf_s = sbase + S::cOff;
  const uint32_t red_s = sbase + S::redOff;
  const uint32_t lred_s = sbase + S::lredOff;
  const uint32_t msm_s = sbase + S::msmOff;
  const uint32_t info_s = sbase + S::infoOff;
  const uint32_t pd_s = sbase + S::pdOff;
  const uint32_t sc_s = sbase + S::scOff;
  const uint32_t stg_s = sbase + S::stgOff;
  const uint32_t ring = sbase + S::ringOff;
  const uint32_t qsm = sbase + S::qOff;
  const uint32_t psm = sbase + S::pOff;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 128);
      mbar_init(&empty[i], 1);
    }
    // 8 rows: the two groups take alternate tiles (one group reads an S
    // buffer, writes a P' buffer); 16 rows: each group owns 8 rows of every tile
    constexpr int SPLIT_READERS = NT == 2 ? 8 : 4;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfull[i], 4);
      mbar_init(&qempty[i], 1 + 4 * NWG);
      mbar_init(&sfull[i], 1);
      mbar_init(&sfree[i], SPLIT_READERS);
      mbar_init(&pfull[i], SPLIT_READERS);
      mbar_init(&pfull[2 + i], SPLIT_READERS);
      mbar_init(&ofull[i], 1);
      mbar_init(&ofull[2 + i], 1);
      mbar_init(&xbar[i], 4);
      mbar_init(&xbar[2 + i], 4);
      mbar_init(&merge[i], NT == 2 ? 4 : 4 * NWG);
      mbar_init(&merge[2 + i], NT == 2 ? 4 : 4 * NWG);
      mbar_init(&mfree[i], 4);
    }
    mbar_init(done, 2);
    *abort_flag = 0;
    *qk_total = -1;
    fence_mbar_init();
  }
  if constexpr (HD < D) {
    // zero the tile ring and the query operands: the dims HD..127 of every row
    // stay zero for the whole launch
    for (int i = threadIdx.x; i < (NS * TILE_BYTES + 2 * S::qBytes) / 16; i += blockDim.x)
      asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(ring + 16 * i), "r"(0u) : "memory");
    fence_proxy_async();
  }
  if (warp == WARP_MMA) tmem_alloc(tmem_slot, S::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int P = p.num_partitions;
  const int Hk = p.num_kv_heads;
  const int RB = p.row_blocks;             // row blocks (virtual heads) per KV head
  const int Hv = Hk * RB;
  const int G = gridDim.x;
  const int QL = EXT ? p.query_len : 1;
  const int rows = EXT ? QL * p.qg : p.qg;   // partial rows per item
  const bool per_token = EXT && p.per_token != 0;
  const int bs = p.block_size;
  const int lbs = p.log2_bs;
  const int bpt = TG / bs;                  // table entries per tile group

  if (warp < WARP_PROD0) {
    // ======================================================== softmax warps
    // Two groups of 4 warps. With 8 query rows group g takes the tiles j with
    // j & 1 == g (buffer b = g) and the groups merge their states per item;
    // with 16 rows (row split) group g owns rows 8g .. 8g + 7 of every tile,
    // reads its 32 columns of S and O and writes its 32 columns of P', and
    // finishes its own rows; its passes take two tiles (P' buffers (j + u) & 3,
    // O buffer = pass & 1). Either way a thread carries RG = 8 rows.
    constexpr int RG = 8;
    constexpr int NG = RS ? 2 : 1;                     // row blocks
    const int wg = warp >> 2;
    const int wq = warp & 3;                           // lane quarter of tensor memory
    const int t = threadIdx.x & 127;                   // tensor-memory lane
    const uint32_t tl = tmem + ((uint32_t)(wq * 32) << 16);
    const float vscale = per_token ? 1.f : __ldg(p.v_scale);
    const int rblk = RS ? wg : 0;                      // this group's row block
    // this token's P' row, the group's 32 columns
    // (PK: the B half's 32 columns follow at + 256)
    const uint32_t ptok = psm + (t >> 3) * (8 * NQS) + (t & 7) * 16 + 256 * rblk;
    // a row's running maximum starts at kNoMax, finite, so that exponent
    // differences stay defined for a row that has seen no token yet (masked
    // scores are -inf: their terms are exactly 0, and two kNoMax give alpha 1)
    constexpr float kNoMax = -1e30f;
    float m[RG], l[RG], o[RG], c[RG];
#pragma unroll
    for (int r = 0; r < RG; ++r) { o[r] = 0.f; m[r] = kNoMax; l[r] = 0.f; c[r] = 0.f; }
    int j = 0, qcnt = 0, pc = 0;         // pc: passes (16 rows)
    bool ok = true;
    int pend_ob = -1;                    // this group's O buffer not folded in yet
    uint32_t pend_oph = 0;               // (its ofull phase)
    // o = (o + O buffer pend_ob) alpha: o and that O are relative to the
    // previous pass's maxima, alpha takes them to the current ones
    auto fold = [&](const float (&alpha)[RG]) -> bool {
      if (!warp_wait(&ofull[pend_ob], pend_oph, abort_flag, KERR_TIMEOUT_FULL)) return false;
      tc_fence_after();
      float w[32];
      // (PK: lanes 64..127, the B half's dims, read the B columns)
      tmem_ld32(tl + 2 * NQK + pend_ob * NQS + 32 * rblk + (PK && wq >= 2 ? NQ : 0), w);
      tmem_wait_ld();
      tc_fence_before();
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        const float sv = fmaf(fmaf(w[2 * RG + r], 0.0625f, w[RG + r]), 0.0625f, w[r]);
        o[r] = fmaf(sv, 0.00390625f, o[r]) * alpha[r];
      }
      return true;
    };

    // the copy warps publish each non-empty item (and a final entry with no
    // tiles) with its query operand
    while (ok) {
      const int qb = qcnt & 1;
      if (!warp_wait(&qfull[qb], (qcnt >> 1) & 1, abort_flag, KERR_TIMEOUT_FULL)) { ok = false; break; }
      const int4 inf = lds_i4(info_s + 32 * qb);
      const int rbase = 16 * lds_i4(info_s + 32 * qb + 16).x;   // the row block's first row
#pragma unroll
      for (int q4 = 0; q4 < RG / 4; ++q4) {
        const float4 cv = lds_f4(cbuf_s + 4 * (qb * R + RG * rblk + 4 * q4));
        c[4 * q4] = cv.x;
        c[4 * q4 + 1] = cv.y;
        c[4 * q4 + 2] = cv.z;
        c[4 * q4 + 3] = cv.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&qempty[qb]);
      const int item = inf.x, L = inf.y, nt = inf.z, tg0 = inf.w;   // tiles of tile groups tg0, tg0 + 1, ...
      if (nt == 0) break;
      // EXT: row qoff * qg + g sees the tokens below L - QL + 1 + qoff; the
      // bound per row, computed once per item (the division by qg is not in
      // the tile loop)
      int vis[RG];
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        m[r] = kNoMax;
        l[r] = 0.f;
        vis[r] = EXT ? L - QL + 1 + (rbase + RG * rblk + r) / p.qg : L;
      }
      // a pass takes NP consecutive tiles of the item (16 rows: two, so that
      // the maxima exchange, the rescale and the O fold run once per 256
      // tokens and the PV of the second tile accumulates onto the first's O;
      // 8 rows: one, every other tile being the other group's)
      for (int i = 0; i < nt;) {
        int np = 1;
        if constexpr (RS) np = min(2, nt - i);
        if (!RS && (j & 1) != wg) {
          ++i;
          ++j;
          continue;
        }
        const int xs = RS ? (pc & 1) : (j & 1);                         // maxima exchange slot
        const uint32_t xph = RS ? (pc >> 1) & 1 : (j >> 1) & 1;
        const int ob = RS ? (pc & 1) : 2 * (j & 1) + ((j >> 1) & 1);    // O buffer (8 rows: also the P' buffer)
        const uint32_t oph = RS ? (pc >> 1) & 1 : (j >> 2) & 1;
        // ---- scores of tile j + u (S buffer (j + u) & 1) into xo
        float x0[RG], x1[RG];
        float vs0 = 1.f, vs1 = 1.f;          // the token's V scale per tile (EXT, per token)
        float xB[PK ? RG : 1];               // PK: the B half's scores (token start + TILE + t)
        auto scores = [&](int u, float (&xo)[RG], float& vso) -> bool {
          const int iu = i + u, ju = j + u, b = ju & 1;
          const int start = PK ? (tg0 + iu) * TG : (tg0 + (iu >> 1)) * TG + (iu & 1) * TILE;
          if (!warp_wait(&sfull[b], (ju >> 1) & 1, abort_flag, KERR_TIMEOUT_FULL)) return false;
          tc_fence_after();
          float v[QT * RG];                  // the row block's S columns: term slot x row
          float vB[PK ? 32 : 1];
          if constexpr (QT == 2) tmem_ld16(tl + b * NQK + 16 * rblk, v);
          else tmem_ld32(tl + b * NQK + 32 * rblk, v);
          if constexpr (PK) tmem_ld32(tl + b * NQK + NQ, vB);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sfree[b]);
          const bool valid = start + t < L;
          // every row sees every token of the tile (warp-uniform): no masks
          const bool whole = start + TILE <= L - (EXT ? QL - 1 : 0);
          float cs[RG];                      // logit multiplier of each row for this token
#pragma unroll
          for (int r = 0; r < RG; ++r) cs[r] = c[r];
          if constexpr (EXT) {
            if (per_token) {
              // the tile's scales landed with its copies (the slot's full barrier)
              if (!warp_wait(&full[ju % NS], (ju / NS) & 1, abort_flag, KERR_TIMEOUT_FULL)) return false;
              const float ks_t = ldsf(sc_s + 4 * ((ju % NS) * 2 * TILE + t));
              vso = valid ? ldsf(sc_s + 4 * ((ju % NS) * 2 * TILE + TILE + t)) : 0.f;
#pragma unroll
              for (int r = 0; r < RG; ++r) cs[r] *= ks_t;
            }
          }
          // the query terms' dot products, T1 + T2/16 (+ T3/256 + T4/4096)
          auto sv_of = [&](int r) -> float {
            if constexpr (QT == 2) return fmaf(v[RG + r], 0.0625f, v[r]);
            else return fmaf(fmaf(fmaf(v[3 * RG + r], 0.0625f, v[2 * RG + r]), 0.0625f, v[RG + r]), 0.0625f, v[r]);
          };
          if (whole) {
#pragma unroll
            for (int r = 0; r < RG; ++r) xo[r] = sv_of(r) * cs[r];
          } else {
#pragma unroll
            for (int r = 0; r < RG; ++r) {
              const float sv = sv_of(r);
              // (EXT: the row's causal bound, which implies start + t < L)
              xo[r] = (EXT ? start + t < vis[r] : valid) ? sv * cs[r] : -INFINITY;
            }
          }
          if constexpr (PK) {
            const bool validB = start + TILE + t < L;
#pragma unroll
            for (int r = 0; r < RG; ++r) {
              const float sv = fmaf(fmaf(fmaf(vB[3 * RG + r], 0.0625f, vB[2 * RG + r]), 0.0625f, vB[RG + r]), 0.0625f,
                                    vB[r]);
              xB[r] = validB ? sv * c[r] : -INFINITY;
            }
          }
          return true;
        };
        if (!scores(0, x0, vs0)) { ok = false; break; }
        if (RS && np > 1) {
          if (!scores(1, x1, vs1)) { ok = false; break; }
        } else {
#pragma unroll
          for (int r = 0; r < RG; ++r) x1[r] = -INFINITY;
        }
        {
          // row maxima over the warp's 32 tokens of the pass (hardware warp reduction)
          float mx[RG];
#pragma unroll
          for (int r = 0; r < RG; ++r) mx[r] = warp_max(PK ? fmaxf(x0[r], xB[r]) : RS ? fmaxf(x0[r], x1[r]) : x0[r]);
          if (lane == 0) {
#pragma unroll
            for (int q4 = 0; q4 < RG / 4; ++q4)
              asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(red_s + 4 * (((xs * NG + rblk) * 4 + wq) * RG + 4 * q4)),
                           "f"(mx[4 * q4]), "f"(mx[4 * q4 + 1]), "f"(mx[4 * q4 + 2]), "f"(mx[4 * q4 + 3]) : "memory");
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&xbar[2 * xs + rblk]);
        if (!warp_wait(&xbar[2 * xs + rblk], xph, abort_flag, KERR_TIMEOUT_FULL)) { ok = false; break; }
        float alpha[RG];
        {
          const uint32_t rb = red_s + (xs * NG + rblk) * 4 * RG * 4;
#pragma unroll
          for (int q4 = 0; q4 < RG / 4; ++q4) {
            const float4 a0 = lds_f4(rb + 16 * q4), a1 = lds_f4(rb + 16 * (RG / 4 + q4));
            const float4 a2 = lds_f4(rb + 16 * (2 * RG / 4 + q4)), a3 = lds_f4(rb + 16 * (3 * RG / 4 + q4));
            const float tm[4] = {fmaxf(fmaxf(a0.x, a1.x), fmaxf(a2.x, a3.x)), fmaxf(fmaxf(a0.y, a1.y), fmaxf(a2.y, a3.y)),
                                 fmaxf(fmaxf(a0.z, a1.z), fmaxf(a2.z, a3.z)), fmaxf(fmaxf(a0.w, a1.w), fmaxf(a2.w, a3.w))};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int r = 4 * q4 + u;
              const float mn = fmaxf(m[r], tm[u]);
              alpha[r] = ex2(m[r] - mn);
              m[r] = mn;
            }
          }
        }
        // ---- probabilities (f16) of a tile's 8 rows for token t, the row sums
        // (first: after the rescale by alpha), and the P' words tw = 3 e4m3
        // terms of 256 p (times the token's V scale, f16, with per-token scales)
        auto split = [&](const float (&xo)[RG], uint32_t vs16, bool first, uint32_t (&tw)[3][RG / 4]) {
#pragma unroll
          for (int k = 0; k < RG / 2; ++k) {
            const uint32_t p16 = f32x2_to_f16x2(ex2(xo[2 * k] - m[2 * k]), ex2(xo[2 * k + 1] - m[2 * k + 1]));
            if (first) {
              l[2 * k] = fmaf(l[2 * k], alpha[2 * k], f16_lo_to_f32(p16));
              l[2 * k + 1] = fmaf(l[2 * k + 1], alpha[2 * k + 1], f16_hi_to_f32(p16));
            } else {
              l[2 * k] += f16_lo_to_f32(p16);
              l[2 * k + 1] += f16_hi_to_f32(p16);
            }
            const uint32_t pv16 = per_token ? hmul2(p16, vs16) : p16;
            uint32_t h = hmul2(pv16, 0x5C005C00u);                     // x 256
            const uint32_t e0 = f16x2_to_e4m3x2(h);
            h = hmul2(hsub2(h, e4m3x2_lo_to_f16x2(e0)), 0x4C004C00u);   // residual x 16
            const uint32_t e1 = f16x2_to_e4m3x2(h);
            h = hmul2(hsub2(h, e4m3x2_lo_to_f16x2(e1)), 0x4C004C00u);
            const uint32_t e2 = f16x2_to_e4m3x2(h);
            if (k & 1) {
              tw[0][k >> 1] = prmt(tw[0][k >> 1], e0, 0x5410u);
              tw[1][k >> 1] = prmt(tw[1][k >> 1], e1, 0x5410u);
              tw[2][k >> 1] = prmt(tw[2][k >> 1], e2, 0x5410u);
            } else {
              tw[0][k >> 1] = e0;
              tw[1][k >> 1] = e1;
              tw[2][k >> 1] = e2;
            }
          }
        };
        // columns slot * 8 + row of the group's 32: terms 0, 1 | term 2, zero slot
        auto store_p = [&](const uint32_t (&tw)[3][RG / 4], uint32_t pb) {
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(pb), "r"(tw[0][0]), "r"(tw[0][1]),
                       "r"(tw[1][0]), "r"(tw[1][1]) : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(pb + 128), "r"(tw[2][0]), "r"(tw[2][1]),
                       "r"(0u), "r"(0u) : "memory");
        };
        // the PV warp's orders for P' buffer pbuf (16 rows): O buffer, accumulate, commit O
        auto order = [&](int pbuf, int u) {
          if (threadIdx.x == 0) {
            const uint32_t d = uint32_t(ob) | (uint32_t(u) << 1) | (uint32_t(u == np - 1) << 2);
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(pd_s + 4 * pbuf), "r"(d) : "memory");
          }
        };
        {
          uint32_t tw0[3][RG / 4];
          split(x0, per_token ? f32x2_to_f16x2(vs0, vs0) : 0u, true, tw0);
          if (RS && np > 1) {
            // both tiles' words at once (independent chains), one proxy fence
            uint32_t tw1[3][RG / 4];
            split(x1, per_token ? f32x2_to_f16x2(vs1, vs1) : 0u, false, tw1);
            store_p(tw0, ptok + (j & 3) * S::pBytes);
            store_p(tw1, ptok + ((j + 1) & 3) * S::pBytes);
            order(j & 3, 0);
            order((j + 1) & 3, 1);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
              mbar_arrive(&pfull[j & 3]);
              mbar_arrive(&pfull[(j + 1) & 3]);
            }
          } else {
            const int pbuf = RS ? j & 3 : ob;
            store_p(tw0, ptok + pbuf * S::pBytes);
            if (RS) order(pbuf, 0);
            if constexpr (PK) {
              // the B half: the same for token start + TILE + t, its columns after A's
              uint32_t twB[3][RG / 4];
              split(xB, 0u, false, twB);
              store_p(twB, ptok + pbuf * S::pBytes + 256);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(&pfull[pbuf]);
          }
        }
        // ---- fold this group's previous O (relative to the previous maxima,
        // so times alpha) while the tensor core computes this pass's
        if (pend_ob >= 0 && !fold(alpha)) { ok = false; break; }
        pend_ob = ob;
        pend_oph = oph;
        i += np;
        j += np;
        ++pc;
      }
      if (ok && pend_ob >= 0) {
        float one[RG];
#pragma unroll
        for (int r = 0; r < RG; ++r) one[r] = 1.f;
        if (!fold(one)) ok = false;
      }
      pend_ob = -1;
      if (!ok) break;

      // ---- item done: row sums over the group's 128 token lanes, then the
      // item's partials. 8 rows: the groups' (m, l, O) merge to a common
      // maximum; the group that does not own the item's last tile merges (it
      // finished first, and with an even tile count per item the owner of the
      // last tile would otherwise always be the same group, which then carries
      // every merge). 16 rows: each group finishes its own 8 rows.
      const uint32_t kph = (qcnt >> 1) & 1;
      const int merger = RS ? wg : (j & 1);
      uint64_t* mbar = &merge[RS ? 2 * qb + wg : qb];
      // (the buffers of item qcnt - 2 must have been read by its merger)
      if (!RS && qcnt >= 2 &&
          !warp_wait(&mfree[qb], ((qcnt >> 1) - 1) & 1, abort_flag, KERR_TIMEOUT_EMPTY)) { ok = false; break; }
      {
        float lr[RG];
#pragma unroll
        for (int r = 0; r < RG; ++r) lr[r] = l[r];
        const float ls = transpose_reduce<RG, false>(lr, lane);
        if ((lane & (32 / RG - 1)) == 0) stsf(lred_s + 4 * ((qb * 4 * NWG + warp) * RG + lane / (32 / RG)), ls);
      }
      if (t == 0) {
#pragma unroll
        for (int r = 0; r < RG; ++r) stsf(msm_s + 4 * ((qb * NWG + wg) * RG + r), m[r]);
      }
      if (!RS && wg != merger) {
#pragma unroll
        for (int r = 0; r < RG; ++r) stsf(stg_s + 4 * ((qb * RG + r) * D + t), o[r]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(mbar);
      if (wg == merger) {
        if (!warp_wait(mbar, kph, abort_flag, KERR_TIMEOUT_FULL)) { ok = false; break; }
        const uint32_t lr = lred_s + qb * 4 * NWG * RG * 4;
        const uint32_t mr = msm_s + qb * NWG * RG * 4;
        const long long row0 = (long long)item * rows + rbase;
        const int rows_here = rows - rbase;
        // [0]: this group, [1]: the other (8 rows only)
        float lsum[2][RG], mg[2][RG];
#pragma unroll
        for (int gi = 0; gi < (RS ? 1 : 2); ++gi) {
          const int g = gi == 0 ? wg : 1 - wg;
#pragma unroll
          for (int q4 = 0; q4 < RG / 4; ++q4) {
            const float4 a0 = lds_f4(lr + 16 * ((4 * g) * RG / 4 + q4)), a1 = lds_f4(lr + 16 * ((4 * g + 1) * RG / 4 + q4));
            const float4 a2 = lds_f4(lr + 16 * ((4 * g + 2) * RG / 4 + q4)), a3 = lds_f4(lr + 16 * ((4 * g + 3) * RG / 4 + q4));
            const float4 mm = lds_f4(mr + 16 * (g * RG / 4 + q4));
            lsum[gi][4 * q4] = (a0.x + a1.x) + (a2.x + a3.x);
            lsum[gi][4 * q4 + 1] = (a0.y + a1.y) + (a2.y + a3.y);
            lsum[gi][4 * q4 + 2] = (a0.z + a1.z) + (a2.z + a3.z);
            lsum[gi][4 * q4 + 3] = (a0.w + a1.w) + (a2.w + a3.w);
            mg[gi][4 * q4] = mm.x;
            mg[gi][4 * q4 + 1] = mm.y;
            mg[gi][4 * q4 + 2] = mm.z;
            mg[gi][4 * q4 + 3] = mm.w;
          }
        }
        float lt_mine = 0.f, mt_mine = 0.f;
#pragma unroll
        for (int r = 0; r < RG; ++r) {
          float mt = mg[0][r], lt = lsum[0][r], ot = o[r];
          if constexpr (!RS) {
            // (a group that saw no token of the item kept kNoMax: its factor is 0
            // next to the other's maximum, 1 with l = 0 when neither saw one)
            const float other = ldsf(stg_s + 4 * ((qb * RG + r) * D + t));
            const float m_me = mg[0][r], m_ot = mg[1][r];
            mt = fmaxf(m_me, m_ot);
            const float a0 = ex2(m_me - mt), a1 = ex2(m_ot - mt);
            lt = lsum[0][r] * a0 + lsum[1][r] * a1;
            ot = o[r] * a0 + other * a1;
          }
          // (lt >= 1: the row maximum's own term is exactly 1; EXT: lt = 0 for a
          // row that saw no token)
          const int row = RG * rblk + r;
          if (row < rows_here && t < PD)
            p.part_o[(row0 + row) * PD + t] = (EXT && lt == 0.f) ? 0.f : ot * (vscale * rcp_approx(lt));
          if (t == r) {
            lt_mine = lt;
            mt_mine = mt;
          }
        }
        if (t < RG && RG * rblk + t < rows_here) {
          // (EXT: a row that saw no token has l = 0 and no maximum)
          p.part_m[row0 + RG * rblk + t] = lt_mine == 0.f ? -INFINITY : mt_mine * kLn2;
          p.part_l[row0 + RG * rblk + t] = lt_mine;
        }
        if (!RS) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&mfree[qb]);
        }
      }
#pragma unroll
      for (int r = 0; r < RG; ++r) o[r] = 0.f;
      ++qcnt;
    }
  } else if (warp < WARP_MMA) {
    // ======================================================== copy warps
    const int pw = warp - WARP_PROD0;
    const uint64_t pol = policy_evict_first();
    // copy lanes: CPR 16-byte chunks per token row, RPI rows per instruction;
    // lane = (row lr, chunk cc), row 32 pw + lr + RPI ii, chunk cc ^ (row & 7)
    constexpr int CPR = HD / 16, RPI = 32 / CPR, NII = 32 / RPI;
    const int lr = lane / CPR, cc = lane % CPR;
    const uint32_t doff_e = (uint32_t)((32 * pw + lr) * D + ((cc ^ (lr & 7)) << 4));
    const uint32_t doff_o = (uint32_t)((32 * pw + lr) * D + ((cc ^ ((lr + 4) & 7)) << 4));
    // PK: the B half's chunks 4 .. 7 of the same rows
    const uint32_t doffB_e = (uint32_t)((32 * pw + lr) * D + (((cc + 4) ^ (lr & 7)) << 4));
    const uint32_t doffB_o = (uint32_t)((32 * pw + lr) * D + (((cc + 4) ^ ((lr + 4) & 7)) << 4));
    const size_t head_bytes = size_t(bs) * HD;
    const size_t v_off = size_t(Hk) * head_bytes;
    const size_t blk_bytes = 2 * v_off;
    const int pt = 32 * pw + lane;                  // query-operand thread: row pt >> 4, dims 8 (pt & 15) ..
    const int qrow = pt >> 4, h16 = pt & 15;
    const float base_scale = (per_token ? 1.f : __ldg(p.k_scale)) * p.softmax_scale * kLog2e;
    int j = 0, qcnt = 0;
    bool ok = true;

    auto seq_len = [&](int sq) -> int { return max(0, min(__ldg(p.seq_lens + sq), p.max_blocks * bs)); };
    auto load_q = [&](int seq, int vh, uint4 (&qv)[NT]) {
#pragma unroll
      for (int h = 0; h < NT; ++h) qv[h] = make_uint4(0, 0, 0, 0);
      if (seq < 0) return;
      const int kvh = vh / RB;
#pragma unroll
      for (int h = 0; h < NT; ++h) {
        const int row = 16 * (vh % RB) + qrow + 8 * h;       // EXT: row qoff * qg + g
        const int qoff = EXT ? row / p.qg : 0, g = EXT ? row - qoff * p.qg : row;
        if (row < rows && h16 < HD / 8)
          qv[h] = __ldg(reinterpret_cast<const uint4*>(p.q + seq * p.q_stride_seq + (EXT ? qoff * p.q_stride_tok : 0) +
                                                       (long long)(kvh * p.qg + g) * p.q_stride_head) + h16);
      }
    };
    auto load_entries = [&](int seq, int tg) -> int32_t {
      if (seq < 0) return 0;
      const int e = tg * bpt + lane;
      return (lane < bpt && e < p.max_blocks) ? __ldg(p.block_table + (long long)seq * p.max_blocks + e) : 0;
    };

    // ---- schedule. One KV head's work is its sequences' tile groups in
    // sequence order, W = sum_s ceil(L_s / TG) of them. The CTAs form groups of
    // Hk, one CTA per head, and the NGe groups split W into equal contiguous
    // ranges: the Hk CTAs of a group stream the same pages at the same time,
    // and every CTA gets the same number of tile groups (+-1) in a handful of
    // items. An item is the part of one (sequence, head) inside a range; its
    // softmax state goes to slot c of the (sequence, head), c = its range
    // minus the range of the sequence's first tile group. NGe is bounded so
    // that no sequence meets more than P ranges; with P = 1 sequences stay
    // whole and belong to the range of their first tile group. Slots without
    // an item get (m, l) = (-inf, 0) and no O.
    const int B = p.num_seqs;
    long long W = 0;
    int Tmax = 0, T0 = 0;                // T0: tile groups of sequence lane (kept for the scan below)
    for (int s0 = 0; s0 < B; s0 += 32) {
      const int T = s0 + lane < B ? (seq_len(s0 + lane) + TG - 1) / TG : 0;
      if (s0 == 0) T0 = T;
      W += (long long)__reduce_add_sync(0xffffffffu, (unsigned)T);
      Tmax = max(Tmax, __reduce_max_sync(0xffffffffu, T));
    }
    int NG, g, h_first, h_step;     // over the virtual heads
    if (G >= Hv) {
      NG = G / Hv; g = blockIdx.x / Hv; h_first = blockIdx.x % Hv; h_step = Hv;
    } else {
      NG = 1; g = 0; h_first = blockIdx.x; h_step = G;
    }
    long long NGe = NG;
    if (P >= 2 && W > 0) {
      // ranges of at least ceil(Tmax / max(1, P - 2)) tile groups: a sequence of
      // T <= Tmax tile groups then meets at most P of them
      const int den = max(1, P - 2);
      const long long rreq = (Tmax + den - 1) / den;
      NGe = max(1LL, min((long long)NG, div_nonneg(W, rreq)));
    }
    const bool active = W > 0 && g < NGe;
    const long long rs = active ? div_nonneg(W * g, NGe) : 0, re = active ? div_nonneg(W * (g + 1), NGe) : 0;
    auto range_of = [&](long long x) -> long long { return div_nonneg((x + 1) * NGe + W - 1, W) - 1; };

    // first sequence of the range: P >= 2, the one holding tile group rs;
    // P = 1, the first one starting at or after rs
    int s_first = B;
    long long off_first = 0;
    if (active) {
      long long base = 0;
      for (int s0 = 0; s0 < B; s0 += 32) {
        const int sq = s0 + lane;
        const int T = s0 == 0 ? T0 : (sq < B ? (seq_len(sq) + TG - 1) / TG : 0);
        int incl = T;
#pragma unroll
        for (int sh = 1; sh < 32; sh <<= 1) {
          const int t2 = __shfl_up_sync(0xffffffffu, incl, sh);
          if (lane >= sh) incl += t2;
        }
        const long long lo = base + incl - T, hi = base + incl;
        const unsigned hit = __ballot_sync(0xffffffffu, sq < B && T > 0 && (P >= 2 ? hi > rs : lo >= rs));
        if (hit) {
          const int src = __ffs(hit) - 1;
          s_first = s0 + src;
          off_first = __shfl_sync(0xffffffffu, lo, src);
          break;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
    }

    // (sequence, head) pairs with no tokens: every slot empty
    for (int pr = blockIdx.x; pr < B * Hk; pr += G) {
      if (seq_len(pr / Hk) == 0) {
        const long long rb = (long long)pr * P * rows;
        for (int i = pt; i < P * rows; i += 128) {
          p.part_m[rb + i] = -INFINITY;
          p.part_l[rb + i] = 0.f;
        }
      }
    }

    // the range's items in order: sequences with tokens whose offset lies
    // below re, then the same walk for the CTA's next head (only when G < Hk)
    struct Cur { int s, h, L; long long off; };
    auto walk = [&](int sq, long long off, int h) -> Cur {
      while (true) {
        while (sq < B && off < re) {
          const int L = seq_len(sq);
          if (L > 0) return Cur{sq, h, L, off};
          ++sq;                                   // no tile groups: the offset stays
        }
        h += h_step;
        if (h >= Hv || s_first >= B) return Cur{-1, h, 0, 0};
        sq = s_first;
        off = off_first;
      }
    };
    auto first_tg = [&](const Cur& c) -> int { return P >= 2 ? (int)(max(rs, c.off) - c.off) : 0; };

    Cur cur = active && s_first < B ? walk(s_first, off_first, h_first) : Cur{-1, 0, 0, 0};
    uint4 qv[NT];
    load_q(cur.s, cur.h, qv);
    int32_t ent0 = load_entries(cur.s, cur.s >= 0 ? first_tg(cur) : 0);
    while (cur.s >= 0 && ok) {
      const int T = (cur.L + TG - 1) / TG;
      int tg_b = 0, tg_e = T, slot = 0, nc = 1;
      if (P >= 2) {
        tg_b = first_tg(cur);
        tg_e = (int)(min(re, cur.off + T) - cur.off);
        const long long r0 = range_of(cur.off);
        slot = (int)(g - r0);
        nc = (int)(range_of(cur.off + T - 1) - r0 + 1);
      }
      const int L = cur.L;
      const int kvh = cur.h / RB;              // the KV head of the virtual head
      const int rblock = cur.h % RB;
      // ring slots of the item: 128-token tiles (the last one dropped when the
      // tile group ends before it), PK: whole tile groups
      const int nt = PK ? tg_e - tg_b : 2 * (tg_e - tg_b) - (((tg_e - 1) * TG + TILE < L) ? 0 : 1);
      const int item = (cur.s * Hk + kvh) * P + slot;
      // next item's query rows and first table entries
      const Cur nxt = walk(cur.s + 1, cur.off + T, cur.h);
      uint4 qn[NT];
      load_q(nxt.s, nxt.h, qn);
      const int32_t ent0n = load_entries(nxt.s, nxt.s >= 0 ? first_tg(nxt) : 0);
      if (slot < 0 || slot >= nc || nc > P || tg_b >= tg_e) {
        // cannot happen with the bound on NGe; never publish a bad slot
        if (lane == 0) atomicExch(&g_kernel_error, KERR_SCHEDULE);
      } else {
        if (slot == 0 && nc < P) {
          const long long rb = ((long long)(cur.s * Hk + kvh) * P + nc) * rows;
          for (int i = pt; i < (P - nc) * rows; i += 128) {
            p.part_m[rb + i] = -INFINITY;
            p.part_l[rb + i] = 0.f;
          }
        }
        // ---- K/V tiles: this warp copies tokens [32 pw, 32 pw + 32) of each;
        // issue_to(n) issues the item's tiles up to n
        const size_t kvh_off = size_t(kvh) * head_bytes;
        int32_t ent = ent0, nent = 0;
        int ti = 0;
        auto issue_to = [&](int i_end) -> bool {
        for (; ti < i_end; ++ti) {
          const int i = ti;
          const int tg = tg_b + (PK ? i : (i >> 1));
          if (PK || (i & 1) == 0) {
            if (i > 0) ent = nent;
            nent = (i + (PK ? 1 : 2) < nt) ? load_entries(cur.s, tg + 1) : 0;
          }
          const int s = j % NS;
          const int rnd = j / NS;
          if (rnd > 0 && !warp_wait(&empty[s], (rnd - 1) & 1, abort_flag, KERR_TIMEOUT_EMPTY)) return false;
          const int tok0 = tg * TG + (PK ? 0 : (i & 1)) * TILE + 32 * pw;
          int pa = __shfl_sync(0xffffffffu, ent, (tok0 & (TG - 1)) >> lbs);
          int pb = __shfl_sync(0xffffffffu, ent, ((tok0 + 16) & (TG - 1)) >> lbs);
          if (pa < 0 || pa >= p.num_blocks) {
            if (tok0 < L && lane == 0) atomicExch(&g_kernel_error, KERR_BAD_BLOCK);
            pa = 0;
          }
          if (pb < 0 || pb >= p.num_blocks) {
            if (tok0 + 16 < L && lane == 0) atomicExch(&g_kernel_error, KERR_BAD_BLOCK);
            pb = 0;
          }
          // tokens tok0 .. tok0 + 15 lie in block pa, tok0 + 16 .. in pb (the same
          // block unless block_size is 16)
          const uint8_t* ka = p.kv + size_t(pa) * blk_bytes + kvh_off + size_t(tok0 & (bs - 1)) * HD + lr * HD + cc * 16;
          const uint8_t* kb = bs == 16 ? p.kv + size_t(pb) * blk_bytes + kvh_off + lr * HD + cc * 16 : ka + 16 * HD;
          const uint32_t slot = ring + s * TILE_BYTES;
#pragma unroll
          for (int ii = 0; ii < NII; ++ii) {
            const bool valid = tok0 + lr + RPI * ii < L;
            const uint8_t* src = ii < NII / 2 ? ka + RPI * HD * ii : kb + RPI * HD * (ii - NII / 2);
            const uint32_t dst = slot + (((RPI * ii) & 4) ? doff_o : doff_e) + RPI * D * ii;
            cp_async16_zfill(dst, src, valid, pol);
            cp_async16_zfill(dst + V_OFF, src + v_off, valid, pol);
          }
          if constexpr (PK) {
            // the B half: tokens tok0 + TILE .., into chunks 4 .. 7 of the same rows
            const int tokB = tok0 + TILE;
            int qa = __shfl_sync(0xffffffffu, ent, (tokB & (TG - 1)) >> lbs);
            int qb2 = __shfl_sync(0xffffffffu, ent, ((tokB + 16) & (TG - 1)) >> lbs);
            if (qa < 0 || qa >= p.num_blocks) {
              if (tokB < L && lane == 0) atomicExch(&g_kernel_error, KERR_BAD_BLOCK);
              qa = 0;
            }
            if (qb2 < 0 || qb2 >= p.num_blocks) {
              if (tokB + 16 < L && lane == 0) atomicExch(&g_kernel_error, KERR_BAD_BLOCK);
              qb2 = 0;
            }
            const uint8_t* kaB = p.kv + size_t(qa) * blk_bytes + kvh_off + size_t(tokB & (bs - 1)) * HD + lr * HD + cc * 16;
            const uint8_t* kbB = bs == 16 ? p.kv + size_t(qb2) * blk_bytes + kvh_off + lr * HD + cc * 16 : kaB + 16 * HD;
#pragma unroll
            for (int ii = 0; ii < NII; ++ii) {
              const bool valid = tokB + lr + RPI * ii < L;
              const uint8_t* src = ii < NII / 2 ? kaB + RPI * HD * ii : kbB + RPI * HD * (ii - NII / 2);
              const uint32_t dst = slot + (((RPI * ii) & 4) ? doffB_o : doffB_e) + RPI * D * ii;
              cp_async16_zfill(dst, src, valid, pol);
              cp_async16_zfill(dst + V_OFF, src + v_off, valid, pol);
            }
          }
          if (per_token && lane < 16) {
            // this warp's 32 tokens' K (lanes 0..7) or V (8..15) scales, 4 tokens
            // per lane; the scale arrays are indexed like the cache's (block, head, slot)
            const int ch = lane & 7;
            const int blk = (bs == 16 && ch >= 4) ? pb : pa;
            const float* sarr = lane < 8 ? p.k_scale : p.v_scale;
            const float* src = sarr + (size_t(blk) * Hk + kvh) * bs + ((tok0 + 4 * ch) & (bs - 1));
            const uint32_t dst = sc_s + 4 * (s * 2 * TILE + (lane < 8 ? 0 : TILE) + 32 * pw + 4 * ch);
            cp_async16_zfill(dst, src, tok0 + 4 * ch < L, pol);
          }
          // the slot's barrier counts this lane once all its copies so far have landed
          // (the timeout test withholds copy warp 0's arrival on the CTA's first tile)
          if (!((p.test_flags & QPA_TEST_WITHHOLD_ARRIVAL) && j == 0 && pw == 0)) cp_async_arrive_noinc(&full[s]);
          ++j;
        }
        return true;
        };
        // a CTA's first item: every ring slot is free, so its first tile goes
        // out before its query operand is built (its copies overlap the build)
        if (qcnt == 0 && !issue_to(1)) {
          ok = false;
          break;
        }
        // ---- query operand: QT e4m3 terms of q 2^a (a per row: max |q| 2^a in [128, 256)),
        // each the rounding of the previous residual times 16 (QT = 4; 2 with 16 rows)
        const int qb = qcnt & 1;
        if (qcnt >= 2 && !warp_wait(&qempty[qb], ((qcnt >> 1) - 1) & 1, abort_flag, KERR_TIMEOUT_EMPTY)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int h = 0; h < NT; ++h) {
          const int row = qrow + 8 * h;
          const uint32_t ws[4] = {qv[h].x, qv[h].y, qv[h].z, qv[h].w};
          float x[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            x[2 * k] = __uint_as_float(ws[k] << 16);
            x[2 * k + 1] = __uint_as_float(ws[k] & 0xffff0000u);
          }
          float amax = 0.f;
#pragma unroll
          for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(x[k]));
#pragma unroll
          for (int sh = 1; sh < 16; sh <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, sh));
          int a = 0;
          if (amax > 0.f) {
            int ex;
            frexpf(amax, &ex);
            a = max(-126, min(126, 8 - ex));
          }
          const float up = __uint_as_float(uint32_t(127 + a) << 23);
          const float down = __uint_as_float(uint32_t(127 - a) << 23);   // 1 / up, exact
#pragma unroll
          for (int k = 0; k < 8; ++k) x[k] *= up;
#pragma unroll
          for (int term = 0; term < QT; ++term) {
            uint32_t e[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              e[k] = f32x2_to_e4m3x2(x[2 * k], x[2 * k + 1]);
              if (term < QT - 1) {
                const uint32_t back = e4m3x2_lo_to_f16x2(e[k]);
                x[2 * k] = (x[2 * k] - f16_lo_to_f32(back)) * 16.f;
                x[2 * k + 1] = (x[2 * k + 1] - f16_hi_to_f32(back)) * 16.f;
              }
            }
            const int rr = (row >> 3) * (8 * QT) + term * 8 + (row & 7);   // S column layout (row block, term, row)
            const uint32_t addr = qsm + qb * S::qBytes + rr * D + (((h16 >> 1) ^ (rr & 7)) << 4) + 8 * (h16 & 1);
            if (h16 < HD / 8)
              asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(e[0] | (e[1] << 16)),
                           "r"(e[2] | (e[3] << 16)) : "memory");
            if (PK && h16 < HD / 8) {
              // the B half's copy of the row: rows NQ.. , dims in bytes 64..127
              const uint32_t addrB = qsm + qb * S::qBytes + (rr + NQ) * D + ((((h16 >> 1) + 4) ^ (rr & 7)) << 4) +
                                     8 * (h16 & 1);
              asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addrB), "r"(e[0] | (e[1] << 16)),
                           "r"(e[2] | (e[3] << 16)) : "memory");
            }
          }
          if (h16 == 0) stsf(cbuf_s + 4 * (qb * R + row), 16 * rblock + row < rows ? base_scale * down : 0.f);
        }
        if (pt == 0) {
          sts_i4(info_s + 32 * qb, make_int4(item, L, nt, tg_b));
          sts_i4(info_s + 32 * qb + 16, make_int4(rblock, 0, 0, 0));
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(&qfull[qb]);
        ++qcnt;

        if (!issue_to(nt)) {
          ok = false;
          break;
        }
      }
      cur = nxt;
#pragma unroll
      for (int h = 0; h < NT; ++h) qv[h] = qn[h];
      ent0 = ent0n;
    }
    if (ok) {
      // final entry: no more items
      const int qb = qcnt & 1;
      if (qcnt < 2 || warp_wait(&qempty[qb], ((qcnt >> 1) - 1) & 1, abort_flag, KERR_TIMEOUT_EMPTY)) {
        if (pt == 0) sts_i4(info_s + 32 * qb, make_int4(0, 0, 0, 0));
        __syncwarp();
        if (lane == 0) mbar_arrive(&qfull[qb]);
      }
    }
    cp_async_wait_all();
  } else if (warp == WARP_MMA) {
    // ======================================================== MMA warp
    // S^T = K Q'^T for every tile in ring order (the softmax groups issue their
    // own PV products).
    if (lane == 0) {
      int qk_j = 0, qcnt = 0;
      bool ok = true;
      while (ok) {
        const int qb = qcnt & 1;
        if (!role_wait(&qfull[qb], (qcnt >> 1) & 1, abort_flag, KERR_TIMEOUT_FULL)) break;
        const int nt = lds_i4(info_s + 32 * qb).z;
        ++qcnt;
        if (nt == 0) break;
        const uint32_t qa = qsm + qb * S::qBytes;
        for (int i = 0; i < nt; ++i, ++qk_j) {
          const int s = qk_j % NS, b = qk_j & 1;
          if (!role_wait(&full[s], (qk_j / NS) & 1, abort_flag, KERR_TIMEOUT_FULL) ||
              (qk_j >= 2 && !role_wait(&sfree[b], ((qk_j >> 1) - 1) & 1, abort_flag, KERR_TIMEOUT_EMPTY))) {
            ok = false;
            break;
          }
          fence_proxy_async();     // the copied bytes (generic proxy) become visible to the tensor core
          tc_fence_after();
          const uint32_t ka = ring + s * TILE_BYTES;
#pragma unroll
          for (int k = 0; k < (PK ? 4 : HD / 32); ++k)
            mma_e4m3(tmem + b * NQK, umma_desc(ka + 32 * k, 16, 1024, kSwizzle128B),
                     umma_desc(qa + 32 * k, 16, 1024, kSwizzle128B), IDESC_QK, k);
          umma_commit(&sfull[b]);
          if (i == nt - 1) umma_commit(&qempty[qb]);
        }
      }
      *qk_total = qk_j;
      // every issued MMA (this warp's and the PV warp's) must finish before the
      // tensor memory is released
      umma_commit(done);
      if (!mbar_try_wait(done, 0)) {
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(done, 0)) {
          if (globaltimer() - t0 > kWaitLimitNs) {
            atomicExch(&g_kernel_error, KERR_TIMEOUT_FULL);
            break;
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ======================================================== PV warp
    // O^T = V^T P'^T for each tile once its softmax group wrote P' (8 rows: one
    // cursor per buffer parity, so the two groups never wait for each other;
    // 16 rows: tiles in order, into the O buffer of their pass); frees the
    // tile's ring slot.
    if (RS && lane == 0) {
      int jj = 0;
      unsigned long long t_prog = globaltimer();
      while (true) {
        const int total = *qk_total;
        if (total >= 0 && jj >= total) break;
        const int pb = jj & 3;
        // (try_wait: the thread sleeps in the barrier instead of spinning on
        // the issue slots of its sub-partition's softmax warps)
        if (mbar_try_wait(&pfull[pb], (jj >> 2) & 1)) {
          tc_fence_after();
          const uint32_t d = lds32(pd_s + 4 * pb);
          const uint32_t ob = d & 1u, acc = (d >> 1) & 1u;
          const uint32_t va = ring + (jj % NS) * TILE_BYTES + V_OFF;
          const uint32_t pa = psm + pb * S::pBytes;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_e4m3(tmem + 2 * NQK + ob * NQS, umma_desc(va + 4096 * k, 16, 1024, kSwizzle128B),
                     umma_desc(pa + k * 32 * NQS, 8 * NQS, 128, kSwizzleNone), IDESC_PV, acc | uint32_t(k));
          umma_commit(&empty[jj % NS]);
          if (d & 4u) umma_commit(&ofull[ob]);
          ++jj;
          t_prog = globaltimer();
        } else {
          if (*abort_flag) break;
          if (globaltimer() - t_prog > kWaitLimitNs) {
            atomicExch(&g_kernel_error, KERR_TIMEOUT_FULL);
            *abort_flag = 1;
            break;
          }
        }
      }
      umma_commit(done);
    } else if (!RS && lane == 0) {
      int pv_n[2] = {0, 1};
      unsigned long long t_prog = globaltimer();
      while (true) {
        const int total = *qk_total;
        if (total >= 0 && pv_n[0] >= total && pv_n[1] >= total) break;
        bool progressed = false;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const int jj = pv_n[b];
          const int ob = 2 * b + ((jj >> 1) & 1);
          if ((total < 0 || jj < total) && mbar_test_wait(&pfull[ob], (jj >> 2) & 1)) {
            tc_fence_after();
            const uint32_t va = ring + (jj % NS) * TILE_BYTES + V_OFF;
            const uint32_t pa = psm + ob * S::pBytes;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_e4m3(tmem + 2 * NQK + ob * NQS, umma_desc(va + 4096 * k, 16, 1024, kSwizzle128B),
                       umma_desc(pa + k * 32 * NQS, 8 * NQS, 128, kSwizzleNone), IDESC_PV, k);
            umma_commit(&ofull[ob]);
            umma_commit(&empty[jj % NS]);
            pv_n[b] += 2;
            progressed = true;
          }
        }
        if (progressed) {
          t_prog = globaltimer();
        } else {
          if (*abort_flag) break;
          if (globaltimer() - t_prog > kWaitLimitNs) {
            atomicExch(&g_kernel_error, KERR_TIMEOUT_FULL);
            *abort_flag = 1;
            break;
          }
        }
      }
      umma_commit(done);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, S::TMEM_COLS);
  }
}

// Flash-combine of the partitions ([PA] reduce kernel), see combine_row: a
// CTA holds rows_per_cta consecutive query rows (seq, kv_head, r), one thread
// group of threads_per_row each, so that a launch is a few hundred CTAs.
// HALVES: the partial rows hold two halves of the output's HD / 2 dims (the
// packed head_dim 64 kernel), added after the combine.
template <typename OutT, int HD, bool HALVES = false>
__global__ void __launch_bounds__(kCombineMaxThreads)
combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_m,
               const float* __restrict__ part_l, OutT* __restrict__ out, int num_kv_heads, int qg,
               int num_partitions, long long out_stride_seq, long long out_stride_head, int rows_per_cta,
               int threads_per_row) {
  extern __shared__ __align__(16) float sw[];
  const int grp = threadIdx.x / threads_per_row, tid = threadIdx.x - grp * threads_per_row;
  const int row = blockIdx.x * rows_per_cta + grp;   // ((seq * Hk) + kvh) * qg + r
  const int r = row % qg;
  const int sk = row / qg;                    // seq * Hk + kvh
  const int seq = sk / num_kv_heads, kvh = sk % num_kv_heads;
  const int gfl = (int)(combine_smem_bytes(num_partitions, threads_per_row) / sizeof(float)) + HD;
  float* my = sw + grp * gfl;
  float* vec = my + gfl - HD;
  combine_row<HD, kCombineKmax128>(part_o, part_m, part_l, (long long)sk * num_partitions * qg + r, qg,
                                   num_partitions, my, vec, tid, threads_per_row);
  constexpr int DO = HALVES ? HD / 2 : HD;     // output dims
  if (tid < DO / 4) {
    OutT* dst = out + seq * out_stride_seq + (long long)(kvh * qg + r) * out_stride_head + 4 * tid;
    if constexpr (HALVES)
      store4(dst, vec[4 * tid] + vec[DO + 4 * tid], vec[4 * tid + 1] + vec[DO + 4 * tid + 1],
             vec[4 * tid + 2] + vec[DO + 4 * tid + 2], vec[4 * tid + 3] + vec[DO + 4 * tid + 3]);
    else
      store4(dst, vec[4 * tid], vec[4 * tid + 1], vec[4 * tid + 2], vec[4 * tid + 3]);
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
  p.q_stride_tok = 0;
  p.query_len = 1;
  p.per_token = 0;
  p.row_blocks = (a.qg + 15) / 16;
  p.test_flags = a.test_flags;
  const long long items = (long long)a.num_seqs * a.num_kv_heads * p.row_blocks * a.num_partitions;
  if (items <= 0) return cudaSuccess;
  const int grid = (int)std::min<long long>(items, (long long)a.num_sms);
  auto launch = [&](auto kernel, int threads, int smem) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    kernel<<<grid, threads, smem, stream>>>(p);
  };
  if (a.head_dim == 64) {
    if (a.qg <= 8)
      launch(pa_fp8_partition_kernel<1, 64, false>, fp8::Smem<1, false, true>::THREADS, fp8::Smem<1, false, true>::total);
    else launch(pa_fp8_partition_kernel<2, 64, false>, fp8::Smem<2>::THREADS, fp8::Smem<2>::total);
  } else {
    if (a.qg <= 8) launch(pa_fp8_partition_kernel<1, 128, false>, fp8::Smem<1>::THREADS, fp8::Smem<1>::total);
    else launch(pa_fp8_partition_kernel<2, 128, false>, fp8::Smem<2>::THREADS, fp8::Smem<2>::total);
  }
  return cudaGetLastError();
}

// The multi-token / per-token decode on the same kernel (rows = query_len *
// qg <= 64, in blocks of 16; head_dim 64 or 128).
cudaError_t launch_fp8x_partition(const Fp8ExtLaunch& a, cudaStream_t stream) {
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
  p.q_stride_tok = a.q_stride_tok;
  p.query_len = a.query_len;
  p.per_token = a.per_token;
  p.test_flags = 0;
  const int rows = a.query_len * a.qg;
  p.row_blocks = (rows + 15) / 16;
  const long long items = (long long)a.num_seqs * a.num_kv_heads * p.row_blocks * a.num_partitions;
  if (items <= 0) return cudaSuccess;
  const int grid = (int)std::min<long long>(items, (long long)a.num_sms);
  auto launch = [&](auto kernel, int threads, int smem) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    kernel<<<grid, threads, smem, stream>>>(p);
  };
  if (a.head_dim == 64) {
    if (rows <= 8)
      launch(pa_fp8_partition_kernel<1, 64, true>, fp8::Smem<1, true>::THREADS, fp8::Smem<1, true>::total);
    else
      launch(pa_fp8_partition_kernel<2, 64, true>, fp8::Smem<2, true>::THREADS, fp8::Smem<2, true>::total);
  } else {
    if (rows <= 8)
      launch(pa_fp8_partition_kernel<1, 128, true>, fp8::Smem<1, true>::THREADS, fp8::Smem<1, true>::total);
    else
      launch(pa_fp8_partition_kernel<2, 128, true>, fp8::Smem<2, true>::THREADS, fp8::Smem<2, true>::total);
  }
  return cudaGetLastError();
}

template <typename OutT, int HD, bool HALVES = false>
static cudaError_t launch_combine_t(const CombineLaunch& a, OutT* out, cudaStream_t stream) {
  const int threads = combine_threads(HD, kCombineKmax128, a.num_partitions);
  const int rpc = combine_rows_per_cta(a.qg, threads);
  const int grid = a.num_seqs * a.num_kv_heads * (a.qg / rpc);
  const size_t smem = size_t(rpc) * (combine_smem_bytes(a.num_partitions, threads) + HD * sizeof(float));
  if (smem > 40 * 1024)
    cudaFuncSetAttribute(combine_kernel<OutT, HD, HALVES>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads * rpc);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // plain stream order: launched as a programmatic dependent of the partition
  // grid (its CTAs cannot sit beside the partition CTAs) the step took ~5 us more
  return cudaLaunchKernelEx(&cfg, combine_kernel<OutT, HD, HALVES>, a.part_o, a.part_m, a.part_l, out, a.num_kv_heads,
                            a.qg, a.num_partitions, a.out_stride_seq, a.out_stride_head, rpc, threads);
}

cudaError_t launch_combine(const CombineLaunch& a, cudaStream_t stream) {
  if (a.num_seqs * a.num_kv_heads * a.qg <= 0) return cudaSuccess;
  cudaError_t e;
  if (a.d == 64 && a.part_d == 128)
    e = a.out_bf16 ? launch_combine_t<__nv_bfloat16, 128, true>(a, static_cast<__nv_bfloat16*>(a.out), stream)
                   : launch_combine_t<float, 128, true>(a, static_cast<float*>(a.out), stream);
  else if (a.d == 64)
    e = a.out_bf16 ? launch_combine_t<__nv_bfloat16, 64>(a, static_cast<__nv_bfloat16*>(a.out), stream)
                   : launch_combine_t<float, 64>(a, static_cast<float*>(a.out), stream);
  else
    e = a.out_bf16 ? launch_combine_t<__nv_bfloat16, 128>(a, static_cast<__nv_bfloat16*>(a.out), stream)
                   : launch_combine_t<float, 128>(a, static_cast<float*>(a.out), stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qpa
