/*
 * qpa.h -- quantised paged-attention decode for NVIDIA GB300 (sm_103a).
 *
 * A C ABI over hand-written CUDA kernels. Every entry point takes plain
 * pointers and sizes, enqueues its kernels on the caller's stream and returns
 * without synchronising. The caller owns every buffer (inputs, outputs and
 * the workspace that holds per-partition partial results); the library
 * allocates nothing and keeps no state between calls, so a call may be
 * captured in a CUDA graph and made from any host thread.
 *
 * Sources the operations follow (web pages, cited by title and section):
 *   [PA]  ROCm/FlyDSL PR #825, "perf(pa tile): readable tile-programming PA
 *         decode kernel" -- fp8 per-tensor paged decode, its partition split,
 *         the flash-combine reduce kernel and the caller-preallocated
 *         partials used under CUDA-graph capture.
 *   [UQ]  vLLM API docs, vllm/v1/attention/ops/flydsl_kernels/
 *         ultraquant_decode_hd256 (PR 59857) -- the 4-bit head_dim=256 slot
 *         cache with in-kernel Walsh-Hadamard rotation of Q (steps A..G).
 *   [IDX] vLLM API docs, vllm/models/minimax_m3/amd/ops/nvfp4_index_decode/
 *         kernel (PR 59747) -- the paged NVFP4 index scorer.
 *
 * Errors: every call returns QPA_OK (0) or a negative status. Argument
 * problems are found on the host before anything is enqueued (no device data
 * is read on the host). QPA_ERR_CUDA reports a launch error from the CUDA
 * runtime. A kernel that meets an invalid block id (outside
 * [0, num_blocks)) reads block 0 instead and raises a device error word;
 * qpa_kernel_error() reads it.
 */
#ifndef QPA_H
#define QPA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QPA_OK 0
#define QPA_ERR_NULL (-1)        /* a required pointer is NULL */
#define QPA_ERR_SHAPE (-2)       /* unsupported head_dim / group / block size / sizes */
#define QPA_ERR_ALIGN (-3)       /* a pointer or stride breaks the 16-byte rule */
#define QPA_ERR_WORKSPACE (-4)   /* workspace smaller than *_workspace_size() */
#define QPA_ERR_PARTITIONS (-5)  /* num_partitions < 1 */
#define QPA_ERR_CUDA (-6)        /* the CUDA runtime rejected a launch */

#define QPA_OUT_F32 0
#define QPA_OUT_BF16 1

/* Returns a static string naming a status code. */
const char* qpa_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
int qpa_version(void);

/* Synchronises `stream` (a cudaStream_t, NULL = legacy default stream), then
 * returns and clears the device error word of the current device: 0 when no
 * kernel reported a problem, otherwise a positive code (1, 2: a wait gave up
 * after its time limit; 3: an invalid block id was met; 4: the fp8 work split
 * produced an out-of-range slot, which its own bounds rule out; 5: a value
 * outside what the hd256 kernel represents, see QPA_UQ_UE8M0_SCALES and the
 * centroid table). Returns QPA_ERR_CUDA
 * if the synchronisation fails. Diagnostic only; the decode entry points
 * never call it. */
int qpa_kernel_error(void* stream);

/* ========================================================================
 * fp8 paged-attention decode ([PA]; 256-token tile groups from [UQ] step F)
 *
 * For every sequence s (length L = seq_lens[s]), KV head h and query row g
 * (query head h*query_group + g):
 *     out = sum_t softmax_t(softmax_scale * q . k_t) v_t,   t = 0 .. L-1,
 *     k_t = e4m3fn(K byte) * (*k_scale),  v_t = e4m3fn(V byte) * (*v_scale).
 * The sequence is split into runs of consecutive 256-token tile groups, at
 * most num_partitions (P) per (s, h); run c writes its softmax state
 * (m_c, l_c, O_c) to slot c of the workspace, the slots after the last run
 * are marked empty (m = -inf, l = 0, O not written), and the combine kernel
 * merges the slots. The runs follow an even split of all sequences' tile
 * groups over the GPU's SMs, so a short sequence usually takes one slot and
 * a long one a few. Any P >= 1 gives the same result (up to rounding).
 * L = 0 gives 0.
 * Precision: the K and V bytes enter the tensor core as they are; each query
 * row, scaled by a power of two, enters as 4 e4m3 terms of its bf16 value (2
 * terms when a KV head has more than 8 query rows), exact for every element
 * down to 2^-22 (2 terms: 2^-14) of the row's largest |q| and within 2^-29
 * (2^-21) of it below; the probabilities enter as the 3 exact e4m3 terms of
 * their f16 value; products accumulate in f32.
 *
 * Layouts (row-major, element counts in brackets):
 *   q           bf16  [num_seqs][num_kv_heads*query_group][128] with the
 *               strides of the descriptor (elements; a multiple of 8), so a
 *               slice of a fused QKV projection can be passed directly.
 *   kv_cache    uint8 [num_blocks][2 (K, V)][num_kv_heads][block_size][128]
 *               e4m3fn bytes; each (block, K/V, head) chunk is contiguous.
 *   block_table int32 [num_seqs][max_blocks_per_seq]; token t of sequence s
 *               is slot t % block_size of block block_table[s][t/block_size].
 *               Only entries below ceil(L/block_size) are read.
 *   seq_lens    int32 [num_seqs]; values are clamped to
 *               [0, max_blocks_per_seq*block_size] on the device.
 *   k_scale,    float [1] each, on the device (read by the kernels).
 *   v_scale
 *   out         [num_seqs][num_kv_heads*query_group][128], float32 or bf16
 *               per out_dtype, contiguous.
 *   workspace   device memory of pa_decode_fp8_workspace_size() bytes,
 *               256-byte aligned; its contents need no initialisation. It
 *               holds, at 256-byte-aligned offsets, float32
 *               O [num_seqs][num_kv_heads][P][query_group][128],
 *               m [num_seqs][num_kv_heads][P][query_group] (max scaled logit,
 *               natural-log units, -inf for an empty slot) and
 *               l [num_seqs][num_kv_heads][P][query_group]
 *               (sum of exp(logit - m), 0 for an empty slot); O is
 *               normalised by l and already multiplied by v_scale. The
 *               combine reads O only where l > 0 and m > -inf.
 * Supported: head_dim 64 or 128 ([PA]), query_group 1..64 (the page's wide
 * GQA; above 16 the kernel runs blocks of 16 query rows of a KV head as
 * separate work streams over the same pages), block_size 16/32/64/128/256.
 * Layouts above with head_dim in place of 128, except the workspace's O for
 * head_dim 64 with query_group <= 8: its rows keep 128 floats, two 64-dim
 * halves (the kernel takes a 256-token tile group per pass as two halves of
 * 128 tokens) that the combine adds.
 * Alignment: q, kv_cache and out 16-byte aligned.
 * ====================================================================== */
typedef struct qpa_fp8_desc {
  int32_t num_seqs;
  int32_t num_kv_heads;
  int32_t query_group;
  int32_t head_dim;
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t out_dtype;        /* QPA_OUT_F32 or QPA_OUT_BF16 */
  int64_t q_stride_seq;     /* elements; 0 = num_kv_heads*query_group*head_dim */
  int64_t q_stride_head;    /* elements; 0 = head_dim */
  float softmax_scale;      /* 0 = 1/sqrt(head_dim) */
  int32_t test_flags;       /* 0; QPA_TEST_WITHHOLD_ARRIVAL only in tests of the timeout path */
} qpa_fp8_desc;

/* Test-only: the partition kernel's first copy warp withholds its arrival on
 * the barrier of its CTA's first K/V tile, so that the roles waiting for that
 * tile run into their time limit. The call returns, the tile's partials are
 * not defined, and qpa_kernel_error() reports 1 or 2. Exercises the bounded
 * waits and the teardown that follows a timeout; not for use otherwise. */
#define QPA_TEST_WITHHOLD_ARRIVAL 1

size_t pa_decode_fp8_workspace_size(const qpa_fp8_desc* d, int num_partitions);

/* Whole decode step: partition kernel then combine kernel, on `stream`. */
int pa_decode_fp8(const void* q, const uint8_t* kv_cache, const int32_t* block_table,
                  const int32_t* seq_lens, const float* k_scale, const float* v_scale,
                  int num_partitions, void* out, const qpa_fp8_desc* d, void* workspace,
                  size_t workspace_bytes, void* stream);

/* The two halves of pa_decode_fp8, for callers that time or schedule them
 * separately. The partition kernel fills the workspace; the combine kernel
 * reads it and writes `out`. */
int pa_decode_fp8_partition(const void* q, const uint8_t* kv_cache, const int32_t* block_table,
                            const int32_t* seq_lens, const float* k_scale, const float* v_scale,
                            int num_partitions, const qpa_fp8_desc* d, void* workspace,
                            size_t workspace_bytes, void* stream);
int pa_decode_fp8_combine(int num_partitions, void* out, const qpa_fp8_desc* d,
                          const void* workspace, size_t workspace_bytes, void* stream);

/* ========================================================================
 * pa_decode_fp8_ext -- fp8 decode of query_len new tokens per sequence
 * (multi-token prediction), with per-tensor or per-token K/V scales
 * ([PA] "per_token_kv" quantisation mode and MTP query_length 1..4 commits).
 *
 * For sequence s (length L = seq_lens[s], counting the query_len new
 * tokens), KV head h, query position qoff in [0, query_len) and group row g
 * (query head h*query_group + g):
 *     out = sum_t softmax_t(softmax_scale * q . k_t) v_t,
 *           t = 0 .. L - query_len + qoff       (causal inside the query block;
 *                                                a row with no token gives 0),
 *     k_t = e4m3fn(K byte) * ks(t),  v_t = e4m3fn(V byte) * vs(t),
 * with ks(t) = k_scale[0] (per-tensor) or the scale of token t's slot
 * (per-token: k_scale[block][h][slot], block and slot of t as for the cache);
 * likewise vs. The per-token layout is this library's reading; the page names
 * the mode only.
 *
 * Layouts: as pa_decode_fp8, except
 *   q         bf16 [num_seqs][query_len][num_kv_heads*query_group][128] with
 *             strides base.q_stride_seq, q_stride_tok and base.q_stride_head
 *             (elements, multiples of 8; 0 selects the contiguous value);
 *   k_scale,  float [1] each (kv_scale_per_token = 0), or float
 *   v_scale   [num_blocks][num_kv_heads][block_size] each, 16-byte aligned
 *             (kv_scale_per_token = 1);
 *   out       [num_seqs][query_len][num_kv_heads*query_group][128], float32
 *             or bf16 per base.out_dtype, contiguous;
 *   workspace pa_decode_fp8_ext_workspace_size() bytes: float32
 *             O [num_seqs][num_kv_heads][P][query_len*query_group][128] and m,
 *             l [num_seqs][num_kv_heads][P][query_len*query_group], row
 *             qoff*query_group + g; O includes the V scale. Slots hold runs
 *             of tile groups as for pa_decode_fp8 (empty slot: m = -inf,
 *             l = 0, O not written); a row that sees no token of a run has
 *             m = -inf, l = 0, O = 0 in that slot.
 * Supported: head_dim 64 or 128, block_size 16..256, query_len 1..4 with
 * query_len * query_group <= 64 (blocks of 16 rows, as for pa_decode_fp8's
 * wide groups). Layouts above with head_dim in place of 128. Errors as
 * pa_decode_fp8; an unsupported query_len or row count is QPA_ERR_SHAPE.
 * ====================================================================== */
typedef struct qpa_fp8_ext_desc {
  qpa_fp8_desc base;
  int32_t query_len;            /* 0 or 1 = one query token */
  int32_t kv_scale_per_token;   /* 0 = per-tensor, 1 = per-token */
  int64_t q_stride_tok;         /* elements; 0 = num_kv_heads*query_group*head_dim */
} qpa_fp8_ext_desc;

size_t pa_decode_fp8_ext_workspace_size(const qpa_fp8_ext_desc* d, int num_partitions);

int pa_decode_fp8_ext(const void* q, const uint8_t* kv_cache, const int32_t* block_table,
                      const int32_t* seq_lens, const float* k_scale, const float* v_scale,
                      int num_partitions, void* out, const qpa_fp8_ext_desc* d, void* workspace,
                      size_t workspace_bytes, void* stream);

/* ========================================================================
 * UltraQuant head_dim=256 4-bit decode ([UQ] steps A..G)
 *
 * For every sequence s, KV head h and query row g (query head h*qg + g):
 *     q_r = q R,  R = H_256 / 16 (orthonormal Sylvester-Hadamard, R = R^T = R^-1)
 *     o_r = sum_t softmax_t(softmax_scale * q_r . k_t) v_t,    out = o_r R
 * where k_t, v_t are the stored (rotated-domain) vectors of token t:
 *     k[d] = e2m1(K code d) * e4m3(K scale byte d/32)
 *     v[d] = centroids[V code d] * e4m3(V scale byte d/32)
 * Slot of (token, KV head), padded_slot bytes (>= 272, a multiple of 16):
 *   bytes   0..127  K codes, dim 2i in the low nibble of byte i
 *   bytes 128..135  K scales (e4m3fn), one per 32 dims
 *   bytes 136..263  V codes (same nibble order)
 *   bytes 264..271  V scales (e4m3fn), one per 32 dims
 * Q is rotated inside the partition kernel and the output is rotated back in
 * the combine kernel. Partition p owns the 32-token slices p, p+P, p+2P, ...
 * of each sequence ([UQ] step F strides 256-token tile groups; the finer
 * granule keeps partitions within one slice of each other, and the combined
 * output does not depend on the split); L = 0 gives 0. The kernel splits each
 * partition's slices over J warps (J = 1, 2, 4 or 8, fixed by num_kv_heads and
 * query_group), each of which keeps its own softmax state, so the workspace
 * holds P*J partial slots per (sequence, KV head): float32
 * O [num_seqs][num_kv_heads][P*J][query_group][256] (rotated domain,
 * normalised by l), m and l [num_seqs][num_kv_heads][P*J][query_group] at
 * 256-byte aligned offsets; a slot without tokens has m = -inf, l = 0 and
 * its O is not written. uq_decode_hd256_workspace_size() accounts for J.
 *
 * Layouts:
 *   q          bf16 [num_seqs][num_kv_heads*query_group][256] (not rotated),
 *              descriptor strides in elements (multiples of 8)
 *   kv_cache   uint8 [num_blocks][block_size][num_kv_heads][padded_slot]
 *   centroids  float32 [16] on the device (code -> value)
 *   block_table, seq_lens, out, workspace: as for pa_decode_fp8 (head_dim 256)
 * Supported: head_dim 256, query_group 1..16, block_size 16/32/64/128/256.
 * Alignment: q, kv_cache and out 16-byte aligned; workspace 256-byte aligned.
 *
 * Precision: q_r enters the QK product rounded to f16, the probabilities
 * too; K is exact (the group scale multiplies the f32 partial dot of each
 * 32-dim group). A centroid table other than the e2m1 values is divided by
 * the power of two 2^e that puts its largest |c| in [0.5, 1) and rounded to
 * f16 (relative error 2^-11), then multiplied by the group scale in f16; the
 * output takes 2^e back, so no table or scale magnitude overflows f16. A
 * non-finite centroid raises error word 5.
 *
 * flags (other bits: QPA_ERR_SHAPE):
 *   QPA_UQ_UE8M0_SCALES  K and V scale bytes are UE8M0, the group scale
 *       format of [UQ] STEP C/F: scale = 2^(byte - 127), byte 0 = 0. Every
 *       byte 0..254 is decoded exactly: the K scale multiplies the f32
 *       partial dot of its group, and each token's V scales are split into
 *       the token's largest power of two (carried by the probability operand
 *       and a per-item reference exponent) and 2^(b - max) <= 1 (applied in
 *       f16). The results are float32 values, so inputs whose logits or
 *       outputs lie beyond float32 are outside the supported range; a byte
 *       255 (the OCP encoding's NaN) in a live token, or a logit that is not
 *       a finite float32, raises error word 5.
 *   QPA_UQ_Q_HAIRCUT  the e4m3 query rounding of [UQ] STEP B' (after the
 *       rotation): the rotated query times softmax_scale is rounded to e4m3
 *       (nearest even, saturating at +-448) and the logits are that rounded
 *       query times k_t, with no further scale:
 *           o_r = sum_t softmax_t(e4m3(softmax_scale * q_r) . k_t) v_t
 *       The rotation feeding the rounding is float32 butterfly stages of
 *       strides 1, 2, ..., 128 (x, y) -> (x + y, x - y), then * 1/16.
 *   QPA_UQ_ROT_PERM  the rotation carries the column permutation of [UQ]
 *       STEP B': R is replaced by M with M[:, perm(d)] = R[:, d],
 *           perm(d) = (d & 0x8F) | ((d >> 2) & 0x10) | ((d << 1) & 0x60),
 *       so q_r = q M, the cache holds k M and v M, and out = o_r M^T. (With
 *       the haircut, the butterfly runs on q[perm^-1(m)] at position m, which
 *       gives 16 q M.)
 * ====================================================================== */
#define QPA_UQ_UE8M0_SCALES 1
#define QPA_UQ_Q_HAIRCUT 2
#define QPA_UQ_ROT_PERM 4

typedef struct qpa_uq_desc {
  int32_t num_seqs;
  int32_t num_kv_heads;
  int32_t query_group;
  int32_t head_dim;         /* 256 */
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t padded_slot;      /* bytes per (token, KV head) slot */
  int32_t out_dtype;        /* QPA_OUT_F32 or QPA_OUT_BF16 */
  int32_t flags;            /* 0 or any of QPA_UQ_UE8M0_SCALES | QPA_UQ_Q_HAIRCUT | QPA_UQ_ROT_PERM */
  int64_t q_stride_seq;     /* elements; 0 = num_kv_heads*query_group*256 */
  int64_t q_stride_head;    /* elements; 0 = 256 */
  float softmax_scale;      /* 0 = 1/sqrt(256) */
} qpa_uq_desc;

size_t uq_decode_hd256_workspace_size(const qpa_uq_desc* d, int num_partitions);

int uq_decode_hd256(const void* q, const uint8_t* kv_cache, const float* centroids,
                    const int32_t* block_table, const int32_t* seq_lens, int num_partitions,
                    void* out, const qpa_uq_desc* d, void* workspace, size_t workspace_bytes,
                    void* stream);
int uq_decode_hd256_partition(const void* q, const uint8_t* kv_cache, const float* centroids,
                              const int32_t* block_table, const int32_t* seq_lens,
                              int num_partitions, const qpa_uq_desc* d, void* workspace,
                              size_t workspace_bytes, void* stream);
int uq_decode_hd256_combine(int num_partitions, void* out, const qpa_uq_desc* d,
                            const void* workspace, size_t workspace_bytes, void* stream);

/* ========================================================================
 * NVFP4 paged index scorer ([IDX] compile_score_decode)
 *
 * For request r (length L = seq_lens[r]), query row qoff < query_len, index
 * head h and block b:
 *     k[t][d]   = e2m1(code[t][d]) * e4m3(scale[t][d/16])
 *     dot[t]    = sum_d e4m3(q[r*query_len + qoff][h][d]) * k[t][d]
 *     scores[h][r*query_len + qoff][b] = max{ dot[t] : t in block b, t <= L - query_len + qoff }
 * and -inf when no token of the block is visible. Every column b of
 * [0, num_cols) of every row is written: columns at or past ceil(L/128) get
 * -inf. No scale, weight or activation is applied to the dot.
 *
 * flags (other bits: QPA_ERR_SHAPE):
 *   QPA_IDX_PER_TOKEN  one column per token instead of per block, i.e. the
 *       dots before the page max ([IDX] frag_max reduces them):
 *           scores[h][r*query_len + qoff][t] = dot[t] if t <= L - query_len + qoff
 *       (t < L follows), else -inf, for every t in [0, num_cols).
 *   QPA_IDX_SHARED_PAGES  the same scores, computed page by page as [IDX]'s
 *       launch loop does: for each block position, the pages of a group of
 *       8 consecutive requests are compared, and a page that several of them
 *       map is loaded and dequantised once and scored for each of them. For
 *       requests that share pages (a common prefix); without sharing the
 *       default request-by-request split is faster.
 *
 * Layouts:
 *   q          uint8 (e4m3fn) [num_reqs*query_len][num_heads][128] with byte
 *              strides q_stride_tok / q_stride_head (multiples of 16)
 *   kv_pages   uint8 [num_blocks] pages at page_stride bytes (>= 9216, a
 *              multiple of 16); a page holds 128 tokens: bytes 0..8191 are
 *              the codes (64 per token, dim 2i in the low nibble of byte i),
 *              bytes 8192..9215 the e4m3 scales (8 per token, one per 16 dims)
 *   block_table int32 [num_reqs][max_blocks_per_seq]; only entries below
 *              min(ceil(L/128), num_cols) are read (per token:
 *              min(ceil(L/128), ceil(num_cols/128)))
 *   seq_lens   int32 [num_reqs]
 *   scores     float32 [num_heads][num_reqs*query_len][num_cols] with element
 *              strides s_stride_head / s_stride_row (the last dim contiguous)
 * Supported: head_dim 128, query_len * num_heads <= 16.
 * Alignment: q and kv_pages 16-byte aligned, scores 4-byte aligned.
 * ====================================================================== */
#define QPA_IDX_PER_TOKEN 1
#define QPA_IDX_SHARED_PAGES 2

typedef struct qpa_idx_desc {
  int32_t num_reqs;
  int32_t query_len;
  int32_t num_heads;
  int32_t head_dim;         /* 128 */
  int32_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t num_cols;         /* S: score columns per row (blocks, or tokens with QPA_IDX_PER_TOKEN) */
  int32_t flags;            /* 0 or QPA_IDX_PER_TOKEN */
  int64_t page_stride;      /* bytes; 0 = 9216 */
  int64_t q_stride_tok;     /* bytes; 0 = num_heads*128 */
  int64_t q_stride_head;    /* bytes; 0 = 128 */
  int64_t s_stride_head;    /* elements; 0 = num_reqs*query_len*num_cols */
  int64_t s_stride_row;     /* elements; 0 = num_cols */
} qpa_idx_desc;

int nvfp4_index_score(const uint8_t* q, const uint8_t* kv_pages, const int32_t* block_table,
                      const int32_t* seq_lens, float* scores, const qpa_idx_desc* d, void* stream);

/* ------------------------------------------------------------------------
 * pa_decode_fp8_static -- pa_decode_fp8 without a workspace argument.
 *
 * The source pages describe no counterpart; this is a convenience of this library. It is
 * meant for callers that cannot call cudaMalloc or otherwise obtain device
 * memory: for example a plugin whose host framework hands it only its input
 * and output tensors, with every device allocation owned by the host
 * application's allocator, or a runtime that reserves all device memory up
 * front and forbids allocations on the decode path. This entry point
 * allocates nothing. The partition partials go to one static device array of
 * QPA_FP8_STATIC_SCRATCH_BYTES (8 MiB), which every GPU that loads the library
 * holds until the process exits.
 *
 * Arguments, layouts and results are those of pa_decode_fp8. The partials
 * need num_seqs*num_kv_heads*num_partitions*query_group*130*4 bytes, plus
 * 256-byte padding; a call that needs more than the array returns
 * QPA_ERR_WORKSPACE without launching anything.
 *
 * The array's device address belongs to a CUDA context. The first call in a
 * (device, context) looks it up, with that device current, and caches it;
 * a call in another context (or after cudaDeviceReset made a new primary
 * context) looks it up again. Make that first call before capturing any
 * stream on that device.
 *
 * All calls share the one array and it keeps the last call's contents.
 * Nothing in it needs to start at zero: the partition kernel writes every
 * partial the combine kernel reads. Calls that overlap on the GPU
 * (different streams, or different host threads on one device) race on the
 * array and must be serialised by the caller.
 * ---------------------------------------------------------------------- */
#define QPA_FP8_STATIC_SCRATCH_BYTES (8u << 20)

int pa_decode_fp8_static(const void* q, const uint8_t* kv_cache, const int32_t* block_table,
                         const int32_t* seq_lens, const float* k_scale, const float* v_scale,
                         int num_partitions, void* out, const qpa_fp8_desc* d, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* QPA_H */
