"""Plain float64 CPU oracle for quantised paged-attention decode.

TEST INFRASTRUCTURE. Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import this package; the library's decode
path never does, and it shares no code, table or helper with the CUDA path.

Sources (web pages; cited by title and section):
  [UQ]  vLLM API docs, ``vllm/v1/attention/ops/flydsl_kernels/
        ultraquant_decode_hd256`` (PR 59857): the head_dim=256 4-bit decode
        kernel ``build_ultraquant_decode_hd256_module``, steps A..G.
  [IDX] vLLM API docs, ``vllm/models/minimax_m3/amd/ops/nvfp4_index_decode/
        kernel`` (PR 59747): the NVFP4 paged index scorer
        ``compile_score_decode``.
  [PA]  ROCm/FlyDSL PR #825, "perf(pa tile): readable tile-programming PA
        decode kernel": fp8 per-tensor paged decode, its partition split and
        flash-combine reduce kernel.

Each function states the passage it follows. Everything is computed directly
from its definition in float64 (numpy), dequantising through the block table
into a dense per-(sequence, KV head) K and V and applying softmax over the
logical, un-paged sequence. There is no blocking or fusion beyond that.

Pinning: every function here is checked by ``tests/test_oracle_*.py`` against
values the pages or the formats fix, closed forms and invariants; see the
header of each module for what pins it.
"""
from .formats import decode_bf16, decode_e2m1, decode_e4m3fn, decode_ue8m0, round_e4m3  # noqa: F401
from .attention import (attend, combine_partials, partition_partials, pa_decode_fp8, pa_decode_fp8_ext,  # noqa: F401
                        tile_groups_of_partition)
from .uq import (decode_uq_slots, perm_dest, perm_source, rotate_q_fp32, rotation_matrix,  # noqa: F401
                 uq_decode_hd256, wht_matrix)
from .scorer import nvfp4_index_score, nvfp4_index_score_per_token, nvfp4_token_dots  # noqa: F401
