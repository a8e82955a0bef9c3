// fp8 (e4m3fn) paged-attention decode of query_len new tokens per sequence,
// with per-tensor or per-token K/V scales: the flash-combine kernel. The
// partition kernel is the tcgen05 kernel of pa_fp8.cu in its multi-token
// variant.
//
// What it computes follows the ROCm/FlyDSL PR #825 page (the "per_token_kv"
// quantisation mode and the MTP query_length 1..4 commits): query position
// qoff of a length-L sequence attends to the tokens t <= L - query_len + qoff
// (causal inside the query block; a row with no visible token gives 0). The
// partials hold query_len x query_group rows per (sequence, KV head, slot),
// row qoff * query_group + g; the combine writes out[seq][qoff][head][dim].
#include "common.cuh"
#include "qpa_internal.h"
#include "combine.cuh"

namespace qpa {

// Flash-combine of the partitions ([PA] reduce) of one query row (sequence,
// KV head, query position, group row), see combine_row.
template <typename OutT, int HD>
__global__ void __launch_bounds__(kCombineMaxThreads)
combine_ext_kernel(const float* __restrict__ part_o, const float* __restrict__ part_m,
                   const float* __restrict__ part_l, OutT* __restrict__ out, int num_kv_heads, int qg,
                   int query_len, int num_partitions, long long out_stride_seq, long long out_stride_tok,
                   long long out_stride_head) {
  extern __shared__ __align__(16) float sw[];
  __shared__ __align__(16) float vec[HD];
  pdl_wait_primary();
  const int rows = query_len * qg;
  const int row = blockIdx.x;                 // ((seq * Hk) + kvh) * rows + r
  const int r = row % rows;
  const int sk = row / rows;                  // seq * Hk + kvh
  const int seq = sk / num_kv_heads, kvh = sk % num_kv_heads;
  const int qoff = r / qg, gq = r % qg;
  combine_row<HD, kCombineKmax128>(part_o, part_m, part_l, (long long)sk * num_partitions * rows + r, rows,
                                   num_partitions, sw, vec);
  if (threadIdx.x < HD / 4) {
    const int t = threadIdx.x;
    OutT* dst = out + seq * out_stride_seq + qoff * out_stride_tok + (long long)(kvh * qg + gq) * out_stride_head + 4 * t;
    store4(dst, vec[4 * t], vec[4 * t + 1], vec[4 * t + 2], vec[4 * t + 3]);
  }
}

// ------------------------------------------------------------------ host side
template <typename OutT, int HD>
static cudaError_t launch_fp8x_combine_t(const Fp8ExtCombineLaunch& a, OutT* out, cudaStream_t stream) {
  const int rows = a.query_len * a.qg;
  const int grid = a.num_seqs * a.num_kv_heads * rows;
  const int threads = combine_threads(HD, kCombineKmax128, a.num_partitions);
  const size_t smem = combine_smem_bytes(a.num_partitions, threads);
  if (smem > 40 * 1024)
    cudaFuncSetAttribute(combine_ext_kernel<OutT, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
  return cudaLaunchKernelEx(&cfg, combine_ext_kernel<OutT, HD>, a.part_o, a.part_m, a.part_l, out, a.num_kv_heads,
                            a.qg, a.query_len, a.num_partitions, a.out_stride_seq, a.out_stride_tok,
                            a.out_stride_head);
}

cudaError_t launch_fp8x_combine(const Fp8ExtCombineLaunch& a, cudaStream_t stream) {
  if (a.num_seqs * a.num_kv_heads * a.query_len * a.qg <= 0) return cudaSuccess;
  cudaError_t e;
  if (a.head_dim == 64)
    e = a.out_bf16 ? launch_fp8x_combine_t<__nv_bfloat16, 64>(a, static_cast<__nv_bfloat16*>(a.out), stream)
                   : launch_fp8x_combine_t<float, 64>(a, static_cast<float*>(a.out), stream);
  else
    e = a.out_bf16 ? launch_fp8x_combine_t<__nv_bfloat16, 128>(a, static_cast<__nv_bfloat16*>(a.out), stream)
                   : launch_fp8x_combine_t<float, 128>(a, static_cast<float*>(a.out), stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qpa
