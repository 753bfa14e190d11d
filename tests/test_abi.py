"""C-ABI checks that need no GPU: the library loads, exports every function
that include/paged_attn.h declares, sizes workspaces, and rejects invalid
arguments on the host with the documented status codes before touching any
device state."""
import ctypes
import re
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__._load_build_module().build()
    import mqa_paged_kv_gb300 as pa
    return pa


def _declared_functions():
    with open(os.path.join(ROOT, "include", "paged_attn.h")) as f:
        text = f.read()
    return re.findall(r"PA_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_abi():
    names = set(_declared_functions())
    assert {"paged_attn_decode", "paged_attn_chunked_prefill", "reshape_and_cache",
            "paged_attn_workspace_bytes", "pa_status_string"} <= names


def test_every_declared_symbol_is_exported(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(so, name), name
    assert set(_declared_functions()) == set(lib.EXPORTED)


def test_status_strings(lib):
    for code in range(-9, 1):
        assert lib.status_string(code) != "unknown status"
    assert lib.status_string(-99) == "unknown status"


def test_workspace_sizes(lib):
    a = lib.paged_attn_workspace_bytes(256, 32, 8, 128, 256, 16, 0)
    b = lib.paged_attn_workspace_bytes(256, 32, 8, 128, 256, 16, 1)
    c = lib.paged_attn_workspace_bytes(8, 32, 8, 128, 2048, 16, 0)
    assert a > b > 0 and c > 0
    # automatic splits up to 2048 sequences: equal shares of the key tiles,
    # two partial slots per warp group of a grid of at most 160 CTAs (8
    # groups of G = 4 heads), each G x (128 + 1) floats, whatever the lengths
    slots = 2 * 160 * 8
    assert a >= slots * 4 * 129 * 4 and c >= slots * 4 * 129 * 4
    assert abs(a - c) < 65536
    # G = 32 (MQA): 4 groups per CTA of 32 heads each
    m = lib.paged_attn_workspace_bytes(128, 32, 1, 128, 64, 16, 0)
    assert m >= 2 * 160 * 4 * 32 * 129 * 4
    # fixed splits, or past 2048 sequences, the sorted work list: partials of
    # every (sequence, split), automatic splits capped at 64 per sequence
    d = lib.paged_attn_workspace_bytes(8, 32, 8, 128, 2048, 16, 64)
    e = lib.paged_attn_workspace_bytes(2100, 32, 8, 128, 2048, 16, 0)
    assert d >= 8 * 64 * 32 * 129 * 4
    assert e >= 2100 * 64 * 32 * 129 * 4
    assert lib.paged_attn_chunked_prefill_workspace_bytes(64, 4434, 32, 8, 128, 256, 16, 0) > 0


FAKE = 0x10000  # never dereferenced: every call below fails host validation


def _decode(lib, **kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, mbs=4, ctx=FAKE, scale=0.125, B=2, Hq=8,
                Hkv=2, D=64, bs=16, NB=8, dtype=1, S=0, out=FAKE, ws=FAKE, wsb=1 << 30)
    args.update(kw)
    a = args
    return lib._lib.paged_attn_decode(a["q"], a["k"], a["v"], a["bt"], a["mbs"], a["ctx"],
                                      a["scale"], a["B"], a["Hq"], a["Hkv"], a["D"], a["bs"],
                                      a["NB"], a["dtype"], a["S"], a["out"], a["ws"], a["wsb"],
                                      None)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=2), -3), (dict(D=96), -4), (dict(D=256), -4), (dict(bs=8), -5),
    (dict(bs=24), -5), (dict(bs=512), -5), (dict(Hq=6, Hkv=4), -2), (dict(Hkv=0), -2),
    (dict(Hq=130, Hkv=2), -2), (dict(S=65), -2), (dict(S=-1), -2), (dict(B=-1), -2),
    (dict(scale=float("nan")), -2), (dict(mbs=0), -2), (dict(NB=0), -2),
    (dict(q=None), -1), (dict(out=None), -1), (dict(bt=None), -1),
    (dict(q=FAKE + 8), -8), (dict(k=FAKE + 2), -8),
    (dict(ws=None), -6), (dict(ws=FAKE + 16), -6), (dict(wsb=16), -6),
])
def test_decode_rejects_bad_arguments(lib, kw, code):
    assert _decode(lib, **kw) == code
    assert lib.last_launch_count() == 0


def test_decode_with_no_sequences_is_a_no_op(lib):
    assert _decode(lib, B=0, q=None, out=None) == 0
    assert lib.last_launch_count() == 0


def test_chunked_prefill_rejects_bad_arguments(lib):
    f = lib._lib.paged_attn_chunked_prefill
    base = [FAKE, FAKE, FAKE, FAKE, 4, FAKE, FAKE, 10, 5, 0.125, 2, 8, 2, 128, 16, 8, 1, 0,
            FAKE, FAKE, 1 << 30, None]
    a = list(base); a[5] = None                     # cu_query_lens
    assert f(*a) == -1
    a = list(base); a[7] = -1                       # total_query_tokens
    assert f(*a) == -2
    a = list(base); a[13] = 80                      # head_dim
    assert f(*a) == -4
    a = list(base); a[20] = 64                      # workspace too small
    assert f(*a) == -6


def test_reshape_and_cache_rejects_bad_arguments(lib):
    f = lib._lib.reshape_and_cache
    base = [FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 16, 8, 1, None, None]
    a = list(base); a[10] = 7
    assert f(*a) == -3
    a = list(base); a[7] = 32
    assert f(*a) == -4
    a = list(base); a[4] = None
    assert f(*a) == -1
    a = list(base); a[0] = FAKE + 4
    assert f(*a) == -8
    a = list(base); a[5] = 0
    assert f(*a) == 0


def test_last_cuda_error_starts_clear(lib):
    # Host-side validation failures are not CUDA errors and leave it clear.
    assert lib._lib.pa_last_cuda_error() == 0
    assert lib._lib.pa_last_cuda_error_string() == b"no error"


def test_varlen_prefill_rejects_bad_arguments(lib):
    f = lib._lib.gqa_varlen_prefill
    P = ctypes.c_void_p
    good = dict(Tq=64, Tk=64, maxq=64, scale=0.1, B=1, Hq=32, Hkv=8, D=128, dtype=1)

    def call(**kw):
        a = dict(good, **kw)
        return f(P(16), P(16), P(16), P(16), P(16), a["Tq"], a["Tk"], a["maxq"], a["scale"],
                 a["B"], a["Hq"], a["Hkv"], a["D"], a["dtype"], P(16), P(256), 1 << 20, None)
    assert call(dtype=7) == -3          # PA_ERR_DTYPE
    assert call(D=96) == -4             # PA_ERR_HEADDIM
    assert call(Hkv=5) == -2            # Hq % Hkv
    assert call(scale=0.0) == -2        # scale must be > 0
    assert call(Tk=0) == -2             # keys needed when there are query rows
    assert call(B=0) == 0 and call(Tq=0) == 0   # nothing to do
    assert lib.gqa_varlen_prefill_workspace_bytes(16, 4096, 32, 8, 128) > 0


def test_cta_limit_is_a_host_setting(lib):
    # no device call: the cap is only stored for the next attention call
    lib.pa_limit_next_call_ctas(32)
    lib.pa_limit_next_call_ctas(0)


# The binding rejects, on the host and before any allocation or launch, what
# a raw pointer cannot carry: shapes that disagree, integer widths, element
# types and host (non-CUDA) tensors.  CPU tensors suffice to reach each check.
def _paged_args(B=4, Hq=8, Hkv=2, D=64, NB=16, bs=16, mbs=4, dt=None):
    import torch
    dt = dt or torch.bfloat16
    return dict(q=torch.zeros(B, Hq, D, dtype=dt), k_cache=torch.zeros(NB, Hkv, bs, D, dtype=dt),
                v_cache=torch.zeros(NB, Hkv, bs, D, dtype=dt),
                block_tables=torch.zeros(B, mbs, dtype=torch.int32),
                context_lens=torch.ones(B, dtype=torch.int32))


def _decode_call(lib, a):
    return lib.paged_attn_decode(a["q"], a["k_cache"], a["v_cache"], a["block_tables"],
                                 a["context_lens"], 0.125, out=a.get("out"))


@pytest.mark.parametrize("change,msg", [
    (lambda a, t: a.update(block_tables=a["block_tables"].long()), "int32"),
    (lambda a, t: a.update(context_lens=a["context_lens"].long()), "int32"),
    (lambda a, t: a.update(context_lens=a["context_lens"][:3].clone()), "block_tables"),
    (lambda a, t: a.update(block_tables=a["block_tables"][:3].clone()), "block_tables"),
    (lambda a, t: a.update(q=a["q"][:3].clone()), "one query row"),
    (lambda a, t: a.update(v_cache=a["v_cache"][:8].clone()), "one shape"),
    (lambda a, t: a.update(k_cache=a["k_cache"].half(), v_cache=a["v_cache"].half()), "dtype"),
    (lambda a, t: a.update(out=t.zeros(4, 8, 64, dtype=t.float16)), "out must match"),
    (lambda a, t: a.update(out=t.zeros(4, 8, 32, dtype=t.bfloat16)), "out must match"),
    (lambda a, t: None, "CUDA tensors"),     # valid shapes, but on the host
])
def test_binding_rejects_mismatched_decode_tensors(lib, change, msg):
    import torch
    a = _paged_args()
    change(a, torch)
    with pytest.raises(ValueError, match=msg):
        _decode_call(lib, a)
    assert lib.last_launch_count() == 0


def test_binding_rejects_mismatched_chunked_tensors(lib):
    import torch
    a = _paged_args()
    for cu, msg in ((torch.tensor([0, 1, 2, 3, 4]).long(), "int32"),
                    (torch.tensor([0, 1, 2, 4], dtype=torch.int32), r"\[B \+ 1\]"),
                    (torch.tensor([0, 1, 2, 3, 4], dtype=torch.int32), "CUDA tensors")):
        for f in (lib.paged_attn_chunked_prefill, lib.paged_attn_cross_attention):
            with pytest.raises(ValueError, match=msg):
                f(a["q"], a["k_cache"], a["v_cache"], a["block_tables"], cu,
                  a["context_lens"], 1, 0.125)


def test_binding_rejects_mismatched_cache_write(lib):
    import torch
    k = torch.zeros(5, 2, 64, dtype=torch.bfloat16)
    kc = torch.zeros(16, 2, 16, 64, dtype=torch.bfloat16)
    sm = torch.zeros(5, dtype=torch.int64)
    with pytest.raises(ValueError, match="slot_mapping"):
        lib.reshape_and_cache(k, k.clone(), kc, kc.clone(), sm[:4].clone())
    with pytest.raises(ValueError, match="int64"):
        lib.reshape_and_cache(k, k.clone(), kc, kc.clone(), sm.int())
    with pytest.raises(ValueError, match="dtype"):
        lib.reshape_and_cache(k, k.half(), kc, kc.clone(), sm)
    with pytest.raises(ValueError, match="32-bit"):
        lib.reshape_and_cache(k, k.clone(), kc, kc.clone(), sm,
                              status_word=torch.zeros(1, dtype=torch.int64))
    with pytest.raises(ValueError, match="CUDA tensors"):
        lib.reshape_and_cache(k, k.clone(), kc, kc.clone(), sm)


def test_binding_rejects_mismatched_varlen_tensors(lib):
    import torch
    q = torch.zeros(10, 8, 64, dtype=torch.bfloat16)
    k = torch.zeros(12, 2, 64, dtype=torch.bfloat16)
    cq = torch.tensor([0, 4, 10], dtype=torch.int32)
    ck = torch.tensor([0, 5, 12], dtype=torch.int32)
    with pytest.raises(ValueError, match="int32"):
        lib.gqa_varlen_prefill(q, k, k.clone(), cq.long(), ck, 6, 0.125)
    with pytest.raises(ValueError, match=r"\[B \+ 1\]"):
        lib.gqa_varlen_prefill(q, k, k.clone(), cq, ck[:2].clone(), 6, 0.125)
    with pytest.raises(ValueError, match="k and v"):
        lib.gqa_varlen_prefill(q, k, k[:11].clone(), cq, ck, 6, 0.125)
    with pytest.raises(ValueError, match="dtype"):
        lib.gqa_varlen_prefill(q, k.half(), k.half(), cq, ck, 6, 0.125)
    with pytest.raises(ValueError, match="CUDA tensors"):
        lib.gqa_varlen_prefill(q, k, k.clone(), cq, ck, 6, 0.125)
    with pytest.raises(ValueError, match="CUDA tensors"):
        lib.pa_read_device_status(torch.zeros(256, dtype=torch.uint8))


def _declared_params():
    """Parameter kinds of every PA_API prototype in include/paged_attn.h:
    'ptr' (any pointer or the stream handle), 'int', 'float', 'size_t', 'u64'."""
    with open(os.path.join(ROOT, "include", "paged_attn.h")) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    out = {}
    for m in re.finditer(r"PA_API\s+[\w\s\*]+?\b(\w+)\s*\(([^)]*)\)\s*;", text):
        params = m.group(2).strip()
        kinds = []
        for p in ([] if params in ("", "void") else params.split(",")):
            if "*" in p or "pa_stream_t" in p:
                kinds.append("ptr")
            elif "size_t" in p:
                kinds.append("size_t")
            elif "uint64_t" in p:
                kinds.append("u64")
            elif "float" in p:
                kinds.append("float")
            else:
                kinds.append("int")
        out[m.group(1)] = kinds
    return out


def test_binding_argtypes_match_the_header(lib):
    # a parameter added, dropped or retyped on one side only would shift or
    # reinterpret every later argument
    decl = _declared_params()
    assert set(decl) == set(_declared_functions())
    for name, kinds in decl.items():
        fn = getattr(lib._lib, name)
        assert fn.argtypes is not None, f"{name}: no argtypes in the binding"
        assert len(fn.argtypes) == len(kinds), (name, len(fn.argtypes), len(kinds))
        for i, (t, k) in enumerate(zip(fn.argtypes, kinds)):
            if k == "ptr":
                ok = t is ctypes.c_void_p or t is ctypes.c_char_p or hasattr(t, "_type_") and \
                    issubclass(t, ctypes._Pointer)
            elif k == "size_t":
                ok = t is ctypes.c_size_t
            elif k == "u64":
                ok = t is ctypes.c_uint64
            elif k == "float":
                ok = t is ctypes.c_float
            else:
                ok = t is ctypes.c_int
            assert ok, (name, i, t, k)
