"""Shared helpers of the GPU parity tests: move a workload case to the GPU,
run the step through the C-ABI binding, and compare with the fp64 oracle."""
import numpy as np
import torch

import oracle
import workloads as W


def elem_dtype(case):
    return torch.float16 if case.dtype == W.F16 else torch.bfloat16


def to_dev(a, dtype=None, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(dtype)
    return t.to(device)


def bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class GpuCase:
    """Device copies of one case's inputs."""

    def __init__(self, case, device="cuda"):
        import mqa_paged_kv_gb300 as pa
        self.pa = pa
        self.case = case
        et = elem_dtype(case)
        self.q = to_dev(case.q, et, device)
        self.k_cache = to_dev(case.k_cache, et, device)
        self.v_cache = to_dev(case.v_cache, et, device)
        self.k_new = to_dev(case.k_new, et, device)
        self.v_new = to_dev(case.v_new, et, device)
        self.slot_mapping = to_dev(case.slot_mapping, device=device)
        self.block_tables = to_dev(case.block_tables, device=device)
        self.context_lens = to_dev(case.context_lens, device=device)
        self.cu_query_lens = to_dev(case.cu_query_lens, device=device)
        self.workspace = None

    def write_cache(self):
        if getattr(self.case, "cross", False):  # static encoder cache
            return
        self.pa.reshape_and_cache(self.k_new, self.v_new, self.k_cache, self.v_cache,
                                  self.slot_mapping)

    def attention(self, num_splits=0, out=None, force_chunked=False):
        c, pa = self.case, self.pa
        B, Hq, D = c.num_seqs, c.num_heads, c.head_dim
        if getattr(c, "cross", False):
            nb = pa.paged_attn_chunked_prefill_workspace_bytes(
                B, c.total_query_tokens, Hq, c.num_kv_heads, D, c.max_blocks_per_seq,
                c.block_size, num_splits)
            if self.workspace is None or self.workspace.numel() < nb:
                self.workspace = pa.alloc_workspace(nb, self.q.device)
            return pa.paged_attn_cross_attention(self.q, self.k_cache, self.v_cache,
                                                 self.block_tables, self.cu_query_lens,
                                                 self.context_lens, c.max_query_len, c.scale,
                                                 out=out, num_splits=num_splits,
                                                 workspace=self.workspace)
        if c.is_decode and not force_chunked:
            nb = pa.paged_attn_workspace_bytes(B, Hq, c.num_kv_heads, D,
                                               c.max_blocks_per_seq, c.block_size, num_splits)
        else:
            nb = pa.paged_attn_chunked_prefill_workspace_bytes(
                B, c.total_query_tokens, Hq, c.num_kv_heads, D, c.max_blocks_per_seq,
                c.block_size, num_splits)
        if self.workspace is None or self.workspace.numel() < nb:
            self.workspace = pa.alloc_workspace(nb, self.q.device)
        if c.is_decode and not force_chunked:
            return pa.paged_attn_decode(self.q, self.k_cache, self.v_cache, self.block_tables,
                                        self.context_lens, c.scale, out=out,
                                        num_splits=num_splits, workspace=self.workspace)
        return pa.paged_attn_chunked_prefill(self.q, self.k_cache, self.v_cache,
                                             self.block_tables, self.cu_query_lens,
                                             self.context_lens, c.max_query_len, c.scale,
                                             out=out, num_splits=num_splits,
                                             workspace=self.workspace)

    def status(self):
        return self.pa.pa_read_device_status(self.workspace)


def half_ulp(x, dtype):
    """Half a unit in the last place of the element type at |x| (normal range)."""
    a = np.maximum(np.abs(x), 1e-30)
    e = np.floor(np.log2(a))
    mant = 10 if dtype == W.F16 else 7
    return np.ldexp(0.5, (e - mant).astype(np.int64))


def check_attention(gpu_bits, o64, obits, dtype, max_tol=1e-2, mean_tol=1e-3):
    """The acceptance rule: max |gpu - fp64| <= 1e-2 (elements with
    |o| >= 4 get half an output ulp on top, since rounding alone exceeds
    1e-2 there), and mean |gpu - oracle rounded to the element type| <= 1e-3.
    Returns the statistics."""
    got = oracle.from_bits(gpu_bits, dtype)
    assert np.all(np.isfinite(got)), "non-finite output"
    err = np.abs(got - o64)
    tol = max_tol + np.where(np.abs(o64) >= 4.0, half_ulp(o64, dtype), 0.0)
    bad = err > tol
    mean_r = float(np.mean(np.abs(got - oracle.from_bits(obits, dtype)))) if got.size else 0.0
    stats = dict(max_abs=float(err.max()) if err.size else 0.0,
                 mean_abs=float(err.mean()) if err.size else 0.0,
                 mean_abs_vs_rounded=mean_r, n=int(err.size),
                 exact_frac=float(np.mean(gpu_bits == obits)) if err.size else 1.0)
    assert not bad.any(), f"max-abs violated at {np.argwhere(bad)[:5].tolist()}: {stats}"
    assert mean_r <= mean_tol, stats
    return stats


def run_and_check(case, rows=None, num_splits=0, check_cache=True):
    """Whole step on the GPU vs the oracle; returns (stats, GpuCase, out)."""
    g = GpuCase(case)
    g.write_cache()
    out = g.attention(num_splits=num_splits)
    torch.cuda.synchronize()
    o64, ob, kref, vref = oracle.run_case(case, rows=rows)
    if check_cache:
        assert np.array_equal(bits(g.k_cache), kref), "k_cache differs"
        assert np.array_equal(bits(g.v_cache), vref), "v_cache differs"
    ob_gpu = bits(out)
    if rows is not None:
        ob_gpu = ob_gpu[np.asarray(rows)]
    stats = check_attention(ob_gpu, o64, ob, case.dtype)
    assert g.status() == 0
    return stats, g, out
