// C-ABI layer: argument validation, workspace carving and kernel launches on
// the caller's stream. Nothing here reads device data or synchronises (except
// qpa_kernel_error, a diagnostic).
#include <cmath>
#include <cstring>

#include "qpa.h"
#include "common.cuh"
#include "qpa_internal.h"

namespace qpa {
__device__ int g_kernel_error = 0;

namespace {

int num_sms_current() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------------ fp8
struct Fp8Layout {
  size_t o_off, m_off, l_off, total;
};

bool fp8_shape_ok(const qpa_fp8_desc* d) {
  if (d->num_seqs < 0 || d->num_kv_heads < 1 || d->query_group < 1 || d->query_group > 64) return false;
  if (d->head_dim != 128 && d->head_dim != 64) return false;
  const int bs = d->block_size;
  if (!(bs == 16 || bs == 32 || bs == 64 || bs == 128 || bs == 256)) return false;
  if (d->num_blocks < 1 || d->max_blocks_per_seq < 1) return false;
  if (d->out_dtype != QPA_OUT_F32 && d->out_dtype != QPA_OUT_BF16) return false;
  if ((long long)d->max_blocks_per_seq * bs > 0x7fffffffLL) return false;
  return true;
}

// Floats per partial O row: head_dim 64 with up to 8 query rows runs the
// packed two-half kernel, whose partials keep both 64-dim halves (the combine
// adds them).
int fp8_part_dim(const qpa_fp8_desc* d, bool ext) {
  return (!ext && d->head_dim == 64 && d->query_group <= 8) ? 128 : d->head_dim;
}

Fp8Layout fp8_layout(const qpa_fp8_desc* d, int P, bool ext = false) {
  const size_t rows = size_t(d->num_seqs) * d->num_kv_heads * P * d->query_group;
  Fp8Layout L;
  L.o_off = 0;
  L.m_off = round_up(L.o_off + rows * fp8_part_dim(d, ext) * sizeof(float), 256);
  L.l_off = round_up(L.m_off + rows * sizeof(float), 256);
  L.total = round_up(L.l_off + rows * sizeof(float), 256);
  return L;
}

int fp8_check(const void* q, const uint8_t* kv, const int32_t* bt, const int32_t* sl, const float* ks,
              const float* vs, int P, const qpa_fp8_desc* d, const void* ws, size_t wsb) {
  if (!d) return QPA_ERR_NULL;
  if (!fp8_shape_ok(d)) return QPA_ERR_SHAPE;
  if (P < 1) return QPA_ERR_PARTITIONS;
  if ((long long)d->num_seqs * d->num_kv_heads * P * d->query_group > 0x7fffffffLL) return QPA_ERR_SHAPE;
  if (d->num_seqs == 0) return QPA_OK;
  if (!q || !kv || !bt || !sl || !ks || !vs || !ws) return QPA_ERR_NULL;
  const long long sh = d->q_stride_head ? d->q_stride_head : d->head_dim;
  const long long ss = d->q_stride_seq ? d->q_stride_seq : (long long)d->num_kv_heads * d->query_group * d->head_dim;
  if (sh < 0 || ss < 0 || (sh % 8) || (ss % 8)) return QPA_ERR_ALIGN;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(ws, 256)) return QPA_ERR_ALIGN;
  if (wsb < fp8_layout(d, P).total) return QPA_ERR_WORKSPACE;
  return QPA_OK;
}

// ------------------------------------------------------------------ fp8, extended
int fp8x_query_len(const qpa_fp8_ext_desc* d) { return d->query_len > 1 ? d->query_len : 1; }

bool fp8x_shape_ok(const qpa_fp8_ext_desc* d) {
  if (!fp8_shape_ok(&d->base)) return false;
  if (d->query_len < 0 || d->query_len > 4) return false;
  if (fp8x_query_len(d) * d->base.query_group > 64) return false;
  if (d->kv_scale_per_token != 0 && d->kv_scale_per_token != 1) return false;
  return true;
}

Fp8Layout fp8x_layout(const qpa_fp8_ext_desc* d, int P) {
  qpa_fp8_desc rows = d->base;
  rows.query_group = d->base.query_group * fp8x_query_len(d);   // partial rows per (seq, head, partition)
  return fp8_layout(&rows, P, true);
}

// ------------------------------------------------------------------ uq hd256
bool uq_shape_ok(const qpa_uq_desc* d) {
  if (d->num_seqs < 0 || d->num_kv_heads < 1 || d->query_group < 1 || d->query_group > 16) return false;
  if (d->head_dim != 256) return false;
  const int bs = d->block_size;
  if (!(bs == 16 || bs == 32 || bs == 64 || bs == 128 || bs == 256)) return false;
  if (d->num_blocks < 1 || d->max_blocks_per_seq < 1) return false;
  if (d->padded_slot < 272 || d->padded_slot % 16) return false;
  if (d->out_dtype != QPA_OUT_F32 && d->out_dtype != QPA_OUT_BF16) return false;
  if ((long long)d->max_blocks_per_seq * bs > 0x7fffffffLL) return false;
  if (d->flags & ~(QPA_UQ_UE8M0_SCALES | QPA_UQ_Q_HAIRCUT | QPA_UQ_ROT_PERM)) return false;
  return true;
}

// Partial slots per (sequence, KV head): P times the kernel's slots per item.
int uq_slots(const qpa_uq_desc* d, int P) { return P * uq_plan(d->num_kv_heads, d->query_group).jw; }

Fp8Layout uq_layout(const qpa_uq_desc* d, int P) {
  const size_t rows = size_t(d->num_seqs) * d->num_kv_heads * uq_slots(d, P) * d->query_group;
  Fp8Layout L;
  L.o_off = 0;
  L.m_off = round_up(rows * 256 * sizeof(float), 256);
  L.l_off = round_up(L.m_off + rows * sizeof(float), 256);
  L.total = round_up(L.l_off + rows * sizeof(float), 256);
  return L;
}

int uq_check(const void* q, const uint8_t* kv, const float* cent, const int32_t* bt, const int32_t* sl, int P,
             const qpa_uq_desc* d, const void* ws, size_t wsb) {
  if (!d) return QPA_ERR_NULL;
  if (!uq_shape_ok(d)) return QPA_ERR_SHAPE;
  if (P < 1) return QPA_ERR_PARTITIONS;
  if ((long long)d->num_seqs * d->num_kv_heads * P * 8 * d->query_group > 0x7fffffffLL) return QPA_ERR_SHAPE;
  if (d->num_seqs == 0) return QPA_OK;
  if (!q || !kv || !cent || !bt || !sl || !ws) return QPA_ERR_NULL;
  const long long sh = d->q_stride_head ? d->q_stride_head : 256;
  const long long ss = d->q_stride_seq ? d->q_stride_seq : (long long)d->num_kv_heads * d->query_group * 256;
  if (sh < 0 || ss < 0 || (sh % 8) || (ss % 8)) return QPA_ERR_ALIGN;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(ws, 256) || !aligned(cent, 4)) return QPA_ERR_ALIGN;
  if (wsb < uq_layout(d, P).total) return QPA_ERR_WORKSPACE;
  return QPA_OK;
}

// ------------------------------------------------------------------ nvfp4 scorer
int idx_check(const uint8_t* q, const uint8_t* pages, const int32_t* bt, const int32_t* sl, const float* sc,
              const qpa_idx_desc* d) {
  if (!d) return QPA_ERR_NULL;
  if (d->num_reqs < 0 || d->query_len < 1 || d->num_heads < 1 || d->head_dim != 128) return QPA_ERR_SHAPE;
  if (d->query_len * d->num_heads > 16 || d->num_blocks < 1 || d->max_blocks_per_seq < 1 || d->num_cols < 1)
    return QPA_ERR_SHAPE;
  if ((long long)d->num_reqs * d->query_len > 0x7fffffffLL) return QPA_ERR_SHAPE;
  if (d->flags & ~(QPA_IDX_PER_TOKEN | QPA_IDX_SHARED_PAGES)) return QPA_ERR_SHAPE;
  if (d->num_reqs == 0) return QPA_OK;
  if (!q || !pages || !bt || !sl || !sc) return QPA_ERR_NULL;
  const long long ps = d->page_stride ? d->page_stride : 9216;
  const long long qt = d->q_stride_tok ? d->q_stride_tok : (long long)d->num_heads * 128;
  const long long qh = d->q_stride_head ? d->q_stride_head : 128;
  if (ps < 9216) return QPA_ERR_SHAPE;
  if ((ps % 16) || (qt % 16) || (qh % 16) || qt < 0 || qh < 0) return QPA_ERR_ALIGN;
  if (!aligned(q, 16) || !aligned(pages, 16) || !aligned(sc, 4)) return QPA_ERR_ALIGN;
  return QPA_OK;
}

}  // namespace
}  // namespace qpa

using namespace qpa;

extern "C" {

const char* qpa_status_string(int s) {
  switch (s) {
    case QPA_OK: return "ok";
    case QPA_ERR_NULL: return "null pointer";
    case QPA_ERR_SHAPE: return "unsupported shape";
    case QPA_ERR_ALIGN: return "misaligned pointer or stride";
    case QPA_ERR_WORKSPACE: return "workspace too small";
    case QPA_ERR_PARTITIONS: return "num_partitions must be >= 1";
    case QPA_ERR_CUDA: return "CUDA launch error";
    default: return "unknown status";
  }
}

int qpa_version(void) { return 100; }

int qpa_kernel_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return QPA_ERR_CUDA;
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, qpa::g_kernel_error, sizeof(int)) != cudaSuccess) return QPA_ERR_CUDA;
  if (cudaMemcpyToSymbol(qpa::g_kernel_error, &z, sizeof(int)) != cudaSuccess) return QPA_ERR_CUDA;
  return v;
}

size_t pa_decode_fp8_workspace_size(const qpa_fp8_desc* d, int num_partitions) {
  if (!d || num_partitions < 1 || !fp8_shape_ok(d)) return 0;
  return fp8_layout(d, num_partitions).total;
}

int pa_decode_fp8_partition(const void* q, const uint8_t* kv_cache, const int32_t* block_table,
                            const int32_t* seq_lens, const float* k_scale, const float* v_scale,
                            int num_partitions, const qpa_fp8_desc* d, void* workspace,
                            size_t workspace_bytes, void* stream) {
  int st = fp8_check(q, kv_cache, block_table, seq_lens, k_scale, v_scale, num_partitions, d, workspace,
                     workspace_bytes);
  if (st != QPA_OK || d->num_seqs == 0) return st;
  const Fp8Layout L = fp8_layout(d, num_partitions);
  Fp8Launch a;
  a.q = q;
  a.kv = kv_cache;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.part_o = reinterpret_cast<float*>(ws + L.o_off);
  a.part_m = reinterpret_cast<float*>(ws + L.m_off);
  a.part_l = reinterpret_cast<float*>(ws + L.l_off);
  a.q_stride_head = d->q_stride_head ? d->q_stride_head : d->head_dim;
  a.q_stride_seq = d->q_stride_seq ? d->q_stride_seq : (long long)d->num_kv_heads * d->query_group * d->head_dim;
  a.num_seqs = d->num_seqs;
  a.num_kv_heads = d->num_kv_heads;
  a.qg = d->query_group;
  a.block_size = d->block_size;
  a.num_blocks = d->num_blocks;
  a.max_blocks = d->max_blocks_per_seq;
  a.num_partitions = num_partitions;
  a.softmax_scale = d->softmax_scale != 0.f ? d->softmax_scale : 1.0f / std::sqrt((float)d->head_dim);
  a.head_dim = d->head_dim;
  a.test_flags = d->test_flags;
  a.num_sms = num_sms_current();
  if (a.num_sms <= 0) return QPA_ERR_CUDA;
  return launch_fp8_partition(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? QPA_OK : QPA_ERR_CUDA;
}

int pa_decode_fp8_combine(int num_partitions, void* out, const qpa_fp8_desc* d, const void* workspace,
                          size_t workspace_bytes, void* stream) {
  if (!d) return QPA_ERR_NULL;
  if (!fp8_shape_ok(d)) return QPA_ERR_SHAPE;
  if (num_partitions < 1) return QPA_ERR_PARTITIONS;
  if (d->num_seqs == 0) return QPA_OK;
  if (!out || !workspace) return QPA_ERR_NULL;
  if (!aligned(out, 16) || !aligned(workspace, 256)) return QPA_ERR_ALIGN;
  const Fp8Layout L = fp8_layout(d, num_partitions);
  if (workspace_bytes < L.total) return QPA_ERR_WORKSPACE;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  CombineLaunch c;
  c.part_o = reinterpret_cast<const float*>(ws + L.o_off);
  c.part_m = reinterpret_cast<const float*>(ws + L.m_off);
  c.part_l = reinterpret_cast<const float*>(ws + L.l_off);
  c.out = out;
  c.out_bf16 = d->out_dtype == QPA_OUT_BF16;
  c.num_seqs = d->num_seqs;
  c.num_kv_heads = d->num_kv_heads;
  c.qg = d->query_group;
  c.num_partitions = num_partitions;
  c.d = d->head_dim;
  c.part_d = fp8_part_dim(d, false);
  c.out_stride_head = d->head_dim;
  c.out_stride_seq = (long long)d->num_kv_heads * d->query_group * d->head_dim;
  return launch_combine(c, static_cast<cudaStream_t>(stream)) == cudaSuccess ? QPA_OK : QPA_ERR_CUDA;
}

int pa_decode_fp8(const void* q, const uint8_t* kv_cache, const int32_t* block_table, const int32_t* seq_lens,
                  const float* k_scale, const float* v_scale, int num_partitions, void* out,
                  const qpa_fp8_desc* d, void* workspace, size_t workspace_bytes, void* stream) {
  int st = fp8_check(q, kv_cache, block_table, seq_lens, k_scale, v_scale, num_partitions, d, workspace,
                     workspace_bytes);
  if (st != QPA_OK) return st;
  if (d->num_seqs == 0) return QPA_OK;
  if (!out) return QPA_ERR_NULL;
  if (!aligned(out, 16)) return QPA_ERR_ALIGN;
  st = pa_decode_fp8_partition(q, kv_cache, block_table, seq_lens, k_scale, v_scale, num_partitions, d,
                               workspace, workspace_bytes, stream);
  if (st != QPA_OK) return st;
  return pa_decode_fp8_combine(num_partitions, out, d, workspace, workspace_bytes, stream);
}

size_t pa_decode_fp8_ext_workspace_size(const qpa_fp8_ext_desc* d, int num_partitions) {
  if (!d || num_partitions < 1 || !fp8x_shape_ok(d)) return 0;
  return fp8x_layout(d, num_partitions).total;
}

int pa_decode_fp8_ext(const void* q, const uint8_t* kv_cache, const int32_t* block_table,
                      const int32_t* seq_lens, const float* k_scale, const float* v_scale,
                      int num_partitions, void* out, const qpa_fp8_ext_desc* d, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!d) return QPA_ERR_NULL;
  if (!fp8x_shape_ok(d)) return QPA_ERR_SHAPE;
  const qpa_fp8_desc* b = &d->base;
  const int QL = fp8x_query_len(d);
  if (num_partitions < 1) return QPA_ERR_PARTITIONS;
  if ((long long)b->num_seqs * b->num_kv_heads * num_partitions * b->query_group * QL > 0x7fffffffLL)
    return QPA_ERR_SHAPE;
  if (b->num_seqs == 0) return QPA_OK;
  if (!q || !kv_cache || !block_table || !seq_lens || !k_scale || !v_scale || !workspace || !out)
    return QPA_ERR_NULL;
  const long long hq = (long long)b->num_kv_heads * b->query_group;
  const long long sh = b->q_stride_head ? b->q_stride_head : b->head_dim;
  const long long st = d->q_stride_tok ? d->q_stride_tok : hq * b->head_dim;
  const long long ss = b->q_stride_seq ? b->q_stride_seq : QL * hq * b->head_dim;
  if (sh < 0 || st < 0 || ss < 0 || (sh % 8) || (st % 8) || (ss % 8)) return QPA_ERR_ALIGN;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(workspace, 256) || !aligned(out, 16))
    return QPA_ERR_ALIGN;
  if (d->kv_scale_per_token && (!aligned(k_scale, 16) || !aligned(v_scale, 16))) return QPA_ERR_ALIGN;
  const Fp8Layout L = fp8x_layout(d, num_partitions);
  if (workspace_bytes < L.total) return QPA_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Fp8ExtLaunch a;
  a.q = q;
  a.kv = kv_cache;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.part_o = reinterpret_cast<float*>(ws + L.o_off);
  a.part_m = reinterpret_cast<float*>(ws + L.m_off);
  a.part_l = reinterpret_cast<float*>(ws + L.l_off);
  a.q_stride_seq = ss;
  a.q_stride_tok = st;
  a.q_stride_head = sh;
  a.num_seqs = b->num_seqs;
  a.num_kv_heads = b->num_kv_heads;
  a.qg = b->query_group;
  a.query_len = QL;
  a.per_token = d->kv_scale_per_token;
  a.block_size = b->block_size;
  a.num_blocks = b->num_blocks;
  a.max_blocks = b->max_blocks_per_seq;
  a.num_partitions = num_partitions;
  a.softmax_scale = b->softmax_scale != 0.f ? b->softmax_scale : 1.0f / std::sqrt((float)b->head_dim);
  a.head_dim = b->head_dim;
  a.num_sms = num_sms_current();
  if (a.num_sms <= 0) return QPA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_fp8x_partition(a, s) != cudaSuccess) return QPA_ERR_CUDA;
  Fp8ExtCombineLaunch c;
  c.part_o = a.part_o;
  c.part_m = a.part_m;
  c.part_l = a.part_l;
  c.out = out;
  c.out_bf16 = b->out_dtype == QPA_OUT_BF16;
  c.num_seqs = b->num_seqs;
  c.num_kv_heads = b->num_kv_heads;
  c.qg = b->query_group;
  c.query_len = QL;
  c.num_partitions = num_partitions;
  c.head_dim = b->head_dim;
  c.out_stride_head = b->head_dim;
  c.out_stride_tok = hq * b->head_dim;
  c.out_stride_seq = QL * hq * b->head_dim;
  return launch_fp8x_combine(c, s) == cudaSuccess ? QPA_OK : QPA_ERR_CUDA;
}

size_t uq_decode_hd256_workspace_size(const qpa_uq_desc* d, int num_partitions) {
  if (!d || num_partitions < 1 || !uq_shape_ok(d)) return 0;
  return uq_layout(d, num_partitions).total;
}

int uq_decode_hd256_partition(const void* q, const uint8_t* kv_cache, const float* centroids,
                              const int32_t* block_table, const int32_t* seq_lens, int num_partitions,
                              const qpa_uq_desc* d, void* workspace, size_t workspace_bytes, void* stream) {
  int st = uq_check(q, kv_cache, centroids, block_table, seq_lens, num_partitions, d, workspace, workspace_bytes);
  if (st != QPA_OK || d->num_seqs == 0) return st;
  const Fp8Layout L = uq_layout(d, num_partitions);
  UqLaunch a;
  a.q = q;
  a.kv = kv_cache;
  a.centroids = centroids;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.part_o = reinterpret_cast<float*>(ws + L.o_off);
  a.part_m = reinterpret_cast<float*>(ws + L.m_off);
  a.part_l = reinterpret_cast<float*>(ws + L.l_off);
  a.q_stride_head = d->q_stride_head ? d->q_stride_head : 256;
  a.q_stride_seq = d->q_stride_seq ? d->q_stride_seq : (long long)d->num_kv_heads * d->query_group * 256;
  a.num_seqs = d->num_seqs;
  a.num_kv_heads = d->num_kv_heads;
  a.qg = d->query_group;
  a.block_size = d->block_size;
  a.num_blocks = d->num_blocks;
  a.max_blocks = d->max_blocks_per_seq;
  a.num_partitions = num_partitions;
  a.padded_slot = d->padded_slot;
  a.softmax_scale = d->softmax_scale != 0.f ? d->softmax_scale : 1.0f / 16.0f;
  a.flags = d->flags;
  a.num_sms = num_sms_current();
  if (a.num_sms <= 0) return QPA_ERR_CUDA;
  return launch_uq_partition(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? QPA_OK : QPA_ERR_CUDA;
}

int uq_decode_hd256_combine(int num_partitions, void* out, const qpa_uq_desc* d, const void* workspace,
                            size_t workspace_bytes, void* stream) {
  if (!d) return QPA_ERR_NULL;
  if (!uq_shape_ok(d)) return QPA_ERR_SHAPE;
  if (num_partitions < 1) return QPA_ERR_PARTITIONS;
  if (d->num_seqs == 0) return QPA_OK;
  if (!out || !workspace) return QPA_ERR_NULL;
  if (!aligned(out, 16) || !aligned(workspace, 256)) return QPA_ERR_ALIGN;
  const Fp8Layout L = uq_layout(d, num_partitions);
  if (workspace_bytes < L.total) return QPA_ERR_WORKSPACE;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  CombineLaunch c;
  c.part_o = reinterpret_cast<const float*>(ws + L.o_off);
  c.part_m = reinterpret_cast<const float*>(ws + L.m_off);
  c.part_l = reinterpret_cast<const float*>(ws + L.l_off);
  c.out = out;
  c.out_bf16 = d->out_dtype == QPA_OUT_BF16;
  c.num_seqs = d->num_seqs;
  c.num_kv_heads = d->num_kv_heads;
  c.qg = d->query_group;
  c.num_partitions = uq_slots(d, num_partitions);
  c.d = 256;
  c.out_stride_head = 256;
  c.out_stride_seq = (long long)d->num_kv_heads * d->query_group * 256;
  c.rot_perm = (d->flags & QPA_UQ_ROT_PERM) != 0;
  return launch_uq_combine(c, static_cast<cudaStream_t>(stream)) == cudaSuccess ? QPA_OK : QPA_ERR_CUDA;
}

int uq_decode_hd256(const void* q, const uint8_t* kv_cache, const float* centroids, const int32_t* block_table,
                    const int32_t* seq_lens, int num_partitions, void* out, const qpa_uq_desc* d, void* workspace,
                    size_t workspace_bytes, void* stream) {
  int st = uq_check(q, kv_cache, centroids, block_table, seq_lens, num_partitions, d, workspace, workspace_bytes);
  if (st != QPA_OK) return st;
  if (d->num_seqs == 0) return QPA_OK;
  if (!out) return QPA_ERR_NULL;
  if (!aligned(out, 16)) return QPA_ERR_ALIGN;
  st = uq_decode_hd256_partition(q, kv_cache, centroids, block_table, seq_lens, num_partitions, d, workspace,
                                 workspace_bytes, stream);
  if (st != QPA_OK) return st;
  return uq_decode_hd256_combine(num_partitions, out, d, workspace, workspace_bytes, stream);
}

int nvfp4_index_score(const uint8_t* q, const uint8_t* kv_pages, const int32_t* block_table,
                      const int32_t* seq_lens, float* scores, const qpa_idx_desc* d, void* stream) {
  const int st = idx_check(q, kv_pages, block_table, seq_lens, scores, d);
  if (st != QPA_OK || d->num_reqs == 0) return st;
  IdxLaunch a;
  a.q = q;
  a.pages = kv_pages;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.scores = scores;
  a.page_stride = d->page_stride ? d->page_stride : 9216;
  a.q_stride_tok = d->q_stride_tok ? d->q_stride_tok : (long long)d->num_heads * 128;
  a.q_stride_head = d->q_stride_head ? d->q_stride_head : 128;
  a.s_stride_row = d->s_stride_row ? d->s_stride_row : d->num_cols;
  a.s_stride_head = d->s_stride_head ? d->s_stride_head : (long long)d->num_reqs * d->query_len * a.s_stride_row;
  a.num_reqs = d->num_reqs;
  a.query_len = d->query_len;
  a.num_heads = d->num_heads;
  a.max_blocks = d->max_blocks_per_seq;
  a.num_cols = d->num_cols;
  a.num_blocks = d->num_blocks;
  a.per_token = (d->flags & QPA_IDX_PER_TOKEN) != 0;
  a.shared_pages = (d->flags & QPA_IDX_SHARED_PAGES) != 0;
  a.num_sms = num_sms_current();
  if (a.num_sms <= 0) return QPA_ERR_CUDA;
  return launch_idx_score(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? QPA_OK : QPA_ERR_CUDA;
}

}  // extern "C"
