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

// Flash-combine of the partitions ([PA] reduce) of the query rows (sequence,
// KV head, query position, group row), see combine_row: rows_per_cta
// consecutive rows per CTA, one thread group of threads_per_row each.
template <typename OutT, int HD>
__global__ void __launch_bounds__(kCombineMaxThreads)
combine_ext_kernel(const float* __restrict__ part_o, const float* __restrict__ part_m,
                   const float* __restrict__ part_l, OutT* __restrict__ out, int num_kv_heads, int qg,
                   int query_len, int num_partitions, long long out_stride_seq, long long out_stride_tok,
                   long long out_stride_head, int rows_per_cta, int threads_per_row) {
  extern __shared__ __align__(16) float sw[];
  const int rows = query_len * qg;
  const int grp = threadIdx.x / threads_per_row, tid = threadIdx.x - grp * threads_per_row;
  const int row = blockIdx.x * rows_per_cta + grp;   // ((seq * Hk) + kvh) * rows + r
  const int r = row % rows;
  const int sk = row / rows;                  // seq * Hk + kvh
  const int seq = sk / num_kv_heads, kvh = sk % num_kv_heads;
  const int qoff = r / qg, gq = r % qg;
  const int gfl = (int)(combine_smem_bytes(num_partitions, threads_per_row) / sizeof(float)) + HD;
  float* my = sw + grp * gfl;
  float* vec = my + gfl - HD;
  combine_row<HD, kCombineKmax128>(part_o, part_m, part_l, (long long)sk * num_partitions * rows + r, rows,
                                   num_partitions, my, vec, tid, threads_per_row);
  if (tid < HD / 4) {
    OutT* dst = out + seq * out_stride_seq + qoff * out_stride_tok + (long long)(kvh * qg + gq) * out_stride_head + 4 * tid;
    store4(dst, vec[4 * tid], vec[4 * tid + 1], vec[4 * tid + 2], vec[4 * tid + 3]);
  }
}

// ------------------------------------------------------------------ host side
template <typename OutT, int HD>
static cudaError_t launch_fp8x_combine_t(const Fp8ExtCombineLaunch& a, OutT* out, cudaStream_t stream) {
  const int rows = a.query_len * a.qg;
  const int threads = combine_threads(HD, kCombineKmax128, a.num_partitions);
  const int rpc = combine_rows_per_cta(rows, threads);
  const int grid = a.num_seqs * a.num_kv_heads * (rows / rpc);
  const size_t smem = size_t(rpc) * (combine_smem_bytes(a.num_partitions, threads) + HD * sizeof(float));
  if (smem > 40 * 1024)
    cudaFuncSetAttribute(combine_ext_kernel<OutT, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads * rpc);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // plain stream order: launched as a programmatic dependent of the partition
  // grid (its CTAs cannot sit beside the partition CTAs) the step took ~5 us more
  return cudaLaunchKernelEx(&cfg, combine_ext_kernel<OutT, HD>, a.part_o, a.part_m, a.part_l, out, a.num_kv_heads,
                            a.qg, a.query_len, a.num_partitions, a.out_stride_seq, a.out_stride_tok,
                            a.out_stride_head, rpc, threads);
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
