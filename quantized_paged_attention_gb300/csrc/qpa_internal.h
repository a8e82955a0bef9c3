// Internal launch descriptors shared by the C-ABI layer and the kernels.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda.h>
#include <stdint.h>
#include <algorithm>

namespace qpa {

struct Fp8Launch {
  const void* q;
  const uint8_t* kv;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const float* k_scale;
  const float* v_scale;
  float* part_o;
  float* part_m;
  float* part_l;
  long long q_stride_seq, q_stride_head;
  int num_seqs, num_kv_heads, qg, block_size, num_blocks, max_blocks, num_partitions;
  float softmax_scale;
  int head_dim;     // 64 or 128
  int test_flags;   // QPA_TEST_WITHHOLD_ARRIVAL
  int num_sms;
};

struct Fp8ExtLaunch {
  const void* q;
  const uint8_t* kv;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const float* k_scale;
  const float* v_scale;
  float* part_o;
  float* part_m;
  float* part_l;
  long long q_stride_seq, q_stride_tok, q_stride_head;
  int num_seqs, num_kv_heads, qg, query_len, per_token, block_size, num_blocks, max_blocks, num_partitions;
  float softmax_scale;
  int head_dim;     // 64 or 128
  int num_sms;
};

struct Fp8ExtCombineLaunch {
  const float* part_o;
  const float* part_m;
  const float* part_l;
  void* out;
  int out_bf16;
  int num_seqs, num_kv_heads, qg, query_len, num_partitions;
  int head_dim;     // 64 or 128
  long long out_stride_seq, out_stride_tok, out_stride_head;
};

struct CombineLaunch {
  const float* part_o;
  const float* part_m;
  const float* part_l;
  void* out;
  int out_bf16;
  int num_seqs, num_kv_heads, qg, num_partitions, d;
  long long out_stride_seq, out_stride_head;
  int rot_perm = 0;   // uq only: undo the rotation's column permutation
  int part_d = 0;     // fp8: floats per partial O row (2 d: two halves to add); 0 = d
};

struct UqLaunch {
  const void* q;
  const uint8_t* kv;
  const float* centroids;
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* part_o;
  float* part_m;
  float* part_l;
  long long q_stride_seq, q_stride_head;
  int num_seqs, num_kv_heads, qg, block_size, num_blocks, max_blocks, num_partitions, padded_slot;
  float softmax_scale;
  int flags;        // QPA_UQ_UE8M0_SCALES | QPA_UQ_Q_HAIRCUT | QPA_UQ_ROT_PERM
  int num_sms;
};

// kernel parameters of the scorer kernels
struct IdxParams {
  const uint8_t* q;
  const uint8_t* pages;
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* scores;
  long long page_stride;                  // bytes
  long long q_stride_tok, q_stride_head;  // bytes
  long long s_stride_head, s_stride_row;  // elements
  int num_reqs, query_len, num_heads, max_blocks, num_cols, num_blocks;
  int per_token;    // one column per token instead of the block max
};

struct IdxLaunch {
  const uint8_t* q;
  const uint8_t* pages;
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* scores;
  long long page_stride, q_stride_tok, q_stride_head;   // bytes
  long long s_stride_head, s_stride_row;                // elements
  int num_reqs, query_len, num_heads, max_blocks, num_cols, num_blocks;
  int per_token;    // one column per token (QPA_IDX_PER_TOKEN)
  int shared_pages; // page-major dedup over groups of 8 requests (QPA_IDX_SHARED_PAGES)
  int num_sms;
};

__device__ __forceinline__ void store4(float* dst, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(dst) = make_float4(a, b, c, d);
}
__device__ __forceinline__ void store4(__nv_bfloat16* dst, float a, float b, float c, float d) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  uint2 v;
  v.x = *reinterpret_cast<uint32_t*>(&lo);
  v.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(dst) = v;
}

cudaError_t launch_fp8_partition(const Fp8Launch& a, cudaStream_t stream);
cudaError_t launch_combine(const CombineLaunch& a, cudaStream_t stream);
cudaError_t launch_fp8x_partition(const Fp8ExtLaunch& a, cudaStream_t stream);
cudaError_t launch_fp8x_combine(const Fp8ExtCombineLaunch& a, cudaStream_t stream);
// How the hd256 partition kernel splits a launch: hg KV heads per work item,
// nh 8-row halves of the query group, jw partial slots per item and head
// (the combine merges num_partitions * jw slots per query row), a ring of
// depth stages, smem bytes of dynamic shared memory.
struct UqPlan {
  int hg, nh, jw, depth, smem;
};
UqPlan uq_plan(int num_kv_heads, int query_group);
cudaError_t launch_uq_partition(const UqLaunch& a, cudaStream_t stream);
cudaError_t launch_uq_combine(const CombineLaunch& a, cudaStream_t stream);
cudaError_t launch_idx_score(const IdxLaunch& a, cudaStream_t stream);

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// The driver's tensor-map encoder, looked up once through the runtime (no
// link-time dependency on the driver library); null if the driver lacks it.
EncodeTiledFn encode_tiled();

}  // namespace qpa
