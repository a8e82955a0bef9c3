"""Helpers shared by the GPU parity tests: move a synthetic case to the
device, run the library through its C ABI, and compute the tolerances the
parity bar states (attention: max|err| <= 2e-3 * max|V| of the sequence and
KV head; scores: |err| <= 1e-4 * max(|ref|, mean|ref| of the row))."""
import numpy as np
import torch

import oracle
import quantized_paged_attention_gb300 as qpa

ATT_TOL = 2e-3
SCORE_TOL = 1e-4


def dev():
    return torch.device("cuda:0")


def bf16_tensor(bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


class Fp8Dev:
    def __init__(self, c, device=None):
        device = device or dev()
        self.c = c
        self.q = bf16_tensor(c.q_bits, device)
        self.kv = torch.from_numpy(c.kv_cache).to(device)
        self.bt = torch.from_numpy(c.block_table).to(device)
        self.sl = torch.from_numpy(c.seq_lens).to(device)
        self.ks = torch.tensor([c.k_scale], dtype=torch.float32, device=device)
        self.vs = torch.tensor([c.v_scale], dtype=torch.float32, device=device)

    def desc(self, out_dtype=torch.float32, q=None):
        q = self.q if q is None else q
        return qpa.fp8_desc(q, self.kv, self.bt, self.c.query_group, self.c.softmax_scale, out_dtype)

    def run(self, P, out_dtype=torch.float32, q=None, workspace=None, out=None):
        q = self.q if q is None else q
        desc = self.desc(out_dtype, q)
        if workspace is None:
            workspace = qpa.alloc_workspace(qpa.pa_decode_fp8_workspace_size(desc, P), q.device)
        out = qpa.pa_decode_fp8(q, self.kv, self.bt, self.sl, self.ks, self.vs, P, self.c.query_group,
                                out=out, workspace=workspace, desc=desc)
        torch.cuda.synchronize()
        assert qpa.kernel_error() == 0
        return out, workspace, desc


def fp8_v_absmax(c, s, h):
    L = int(c.seq_lens[s])
    if L == 0:
        return 0.0
    _, v = oracle.attention.dense_kv_fp8(c.kv_cache, c.block_table, s, h, L, c.k_scale, c.v_scale)
    return float(np.abs(v).max())


def check_attention(got, ref, vmax_fn, c, units=None, what=""):
    """got/ref [B, Hq, D]; vmax_fn(s, h) -> max|V| for the tolerance."""
    B = got.shape[0]
    Hk, QG = c.num_kv_heads, c.query_group
    if units is None:
        units = [(s, h) for s in range(B) for h in range(Hk)]
    worst = 0.0
    for s, h in units:
        rows = slice(h * QG, (h + 1) * QG)
        g, r = got[s, rows], ref[s, rows]
        assert np.all(np.isfinite(g)), f"{what} non-finite output at seq {s} head {h}"
        L = int(c.seq_lens[s])
        if L == 0:
            assert np.all(g == 0.0), f"{what} L=0 must give 0 (seq {s})"
            continue
        err = float(np.max(np.abs(g - r)))
        tol = ATT_TOL * vmax_fn(s, h)
        worst = max(worst, err / tol if tol > 0 else 0.0)
        assert err <= tol, f"{what} seq {s} head {h}: max|err| {err:.3e} > tol {tol:.3e}"
    return worst


class UqDev:
    def __init__(self, c, device=None):
        device = device or dev()
        self.c = c
        self.q = bf16_tensor(c.q_bits, device)
        self.kv = torch.from_numpy(c.kv_cache).to(device)
        self.cent = torch.from_numpy(np.ascontiguousarray(c.centroids, dtype=np.float32)).to(device)
        self.bt = torch.from_numpy(c.block_table).to(device)
        self.sl = torch.from_numpy(c.seq_lens).to(device)

    def desc(self, out_dtype=torch.float32, q_haircut=False):
        return qpa.uq_desc(self.q, self.kv, self.bt, self.c.query_group, self.c.softmax_scale, out_dtype,
                           self.c.scale_format, q_haircut, self.c.rot_perm)

    def run(self, P, out_dtype=torch.float32, workspace=None, q_haircut=False):
        desc = self.desc(out_dtype, q_haircut)
        if workspace is None:
            workspace = qpa.alloc_workspace(qpa.uq_decode_hd256_workspace_size(desc, P), self.q.device)
        out = qpa.uq_decode_hd256(self.q, self.kv, self.cent, self.bt, self.sl, P, self.c.query_group,
                                  workspace=workspace, desc=desc)
        torch.cuda.synchronize()
        assert qpa.kernel_error() == 0
        return out, workspace, desc


def uq_v_absmax(c, s, h):
    L = int(c.seq_lens[s])
    if L == 0:
        return 0.0
    _, v = oracle.uq.dense_kv_uq(c.kv_cache, c.centroids, c.block_table, s, h, L, c.scale_format)
    return float(np.abs(v).max())


class IdxDev:
    def __init__(self, c, device=None, stride_pad=0):
        """stride_pad > 0 stores the pages at a stride of 9216 + stride_pad
        bytes (a view into a wider buffer)."""
        device = device or dev()
        self.c = c
        self.q = torch.from_numpy(c.q_codes).to(device)
        pages = torch.from_numpy(c.pages)
        if stride_pad:
            wide = torch.zeros((pages.shape[0], pages.shape[1] + stride_pad), dtype=torch.uint8)
            wide[:, :pages.shape[1]] = pages
            self.pages = wide.to(device)[:, :pages.shape[1]]
        else:
            self.pages = pages.to(device)
        self.bt = torch.from_numpy(c.block_table).to(device)
        self.sl = torch.from_numpy(c.seq_lens).to(device)

    def run(self, scores=None, per_token_cols=None, shared_pages=False):
        """Block scores over c.num_cols columns, or with per_token_cols the
        per-token scores over that many token columns; shared_pages selects
        the page-by-page dedup split."""
        cols = self.c.num_cols if per_token_cols is None else per_token_cols
        out = qpa.nvfp4_index_score(self.q, self.pages, self.bt, self.sl, self.c.query_len, cols,
                                    scores=scores, per_token=per_token_cols is not None, shared_pages=shared_pages)
        torch.cuda.synchronize()
        assert qpa.kernel_error() == 0
        return out


def check_scores(got, ref, rows=None, what=""):
    """got/ref [H, rows, S]: -inf must match exactly; finite values within
    1e-4 * max(|ref|, mean |ref| of the row's finite scores)."""
    if rows is not None:
        got, ref = got[:, rows], ref[:, rows]
    ninf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), ninf), f"{what}: -inf pattern differs"
    assert not np.any(np.isnan(got)), f"{what}: NaN in scores"
    fin = ~ninf
    with np.errstate(invalid="ignore"):
        cnt = fin.sum(axis=2, keepdims=True)
        rowsum = np.where(fin, np.abs(ref), 0.0).sum(axis=2, keepdims=True)
        rowmean = np.where(cnt > 0, rowsum / np.maximum(cnt, 1), 0.0)
        bound = SCORE_TOL * np.maximum(np.abs(ref), rowmean)
        err = np.where(fin, np.abs(got - ref), 0.0)
    bad = fin & (err > bound)
    assert not np.any(bad), f"{what}: {int(bad.sum())} scores out of tolerance, worst {float(np.nanmax(np.where(fin, err / np.maximum(bound, 1e-30), np.nan))):.3g}x"
