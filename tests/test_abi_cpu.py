"""The C ABI without a GPU: the library loads, exports every function the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

from sparse_latent_attention_decode_b300 import mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla_decode.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "return")))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for want in ("rope_freqs_init", "mla_rope_apply", "mla_rope_apply_layout", "mla_absorb_q", "mla_sparse_decode", "mla_out_up",
                 "mla_sparse_decode_workspace_size", "mla_status_string"):
        assert want in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(mla.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert set(mla.EXPORTED) <= set(_declared_functions())


def test_softmax_scale_from_the_library_matches_closed_form():
    g = {}
    for line in open(os.path.join(ROOT, "tests", "golden", "softmax_scale_closed_form.txt")):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            g[k] = float(v)
    assert mla.softmax_scale() == pytest.approx(g["softmax_scale"], rel=1e-15)
    p = mla.rope_params(max_seq_len=4096)
    assert mla.softmax_scale(p) == pytest.approx(g["softmax_scale_no_yarn"], rel=1e-15)


def test_workspace_size_is_monotone_and_rejects_bad_sizes():
    lib = mla._lib
    assert lib.mla_sparse_decode_workspace_size(0, 2048) == 0
    assert lib.mla_sparse_decode_workspace_size(64, 0) == 0
    assert lib.mla_sparse_decode_workspace_size(5000, 16) == 0
    # small batches split the selection over the idle CTA pairs and keep fp32 partials, so
    # the size is not monotone in B below 74 rows; it is in K, and in B once nothing splits
    a = lib.mla_sparse_decode_workspace_size(1, 2048)
    b = lib.mla_sparse_decode_workspace_size(64, 2048)
    c = lib.mla_sparse_decode_workspace_size(64, 16384)
    d = lib.mla_sparse_decode_workspace_size(74, 2048)
    e = lib.mla_sparse_decode_workspace_size(128, 2048)
    assert 0 < a and 0 < b <= c and 0 < d < e
    assert all(x % 256 == 0 for x in (a, b, c, d, e))
    # every batch that splits stays within the fixed workspace of the static entry point
    for B in (1, 2, 3, 5, 16, 37, 73):
        assert lib.mla_sparse_decode_workspace_size(B, 2048) <= mla.STATIC_WS_BYTES


P = ctypes.c_void_p
GOOD = P(0x10000)       # never dereferenced: every call below fails its host check first
MISALIGNED = P(0x10004)


def test_host_argument_checks_return_codes_without_launching():
    lib = mla._lib
    nul = None
    # NULL pointers
    assert lib.mla_sparse_decode(nul, GOOD, GOOD, 16, GOOD, 8, GOOD, 1, 1.0, nul, GOOD, GOOD, 1 << 30, nul,
                                 nul) == -1
    assert lib.mla_absorb_q(GOOD, nul, GOOD, 16, GOOD, GOOD, 1, GOOD, nul, nul) == -1
    assert lib.mla_out_up(GOOD, nul, 1, GOOD, nul) == -1
    assert lib.mla_rope_apply(GOOD, GOOD, 16, nul, 1, GOOD, nul, nul) == -1
    assert lib.rope_freqs_init(nul, ctypes.byref(mla.rope_params()), nul) == -1
    # alignment
    assert lib.mla_out_up(MISALIGNED, GOOD, 1, GOOD, nul) == -2
    assert lib.mla_sparse_decode(GOOD, GOOD, GOOD, 16, GOOD, 8, GOOD, 1, 1.0, nul, GOOD, P(0x10010), 1 << 30,
                                 nul, nul) == -2          # workspace must be 256-byte aligned
    # sizes
    assert lib.mla_sparse_decode(GOOD, GOOD, GOOD, 16, GOOD, 8, GOOD, 0, 1.0, nul, GOOD, GOOD, 1 << 30, nul,
                                 nul) == -3
    assert lib.mla_sparse_decode(GOOD, GOOD, GOOD, 0, GOOD, 8, GOOD, 1, 1.0, nul, GOOD, GOOD, 1 << 30, nul,
                                 nul) == -3
    assert lib.mla_sparse_decode(GOOD, GOOD, GOOD, 16, GOOD, 0, GOOD, 1, 1.0, nul, GOOD, GOOD, 1 << 30, nul,
                                 nul) == -3
    assert lib.mla_absorb_q(GOOD, GOOD, GOOD, 16, GOOD, GOOD, 4097, GOOD, nul, nul) == -3
    assert lib.mla_out_up(GOOD, GOOD, 0, GOOD, nul) == -3
    bad = mla.rope_params()
    bad.rope_dim = 32
    assert lib.rope_freqs_init(GOOD, ctypes.byref(bad), nul) == -3
    bad = mla.rope_params()
    bad.rope_factor = 0.0
    assert lib.rope_freqs_init(GOOD, ctypes.byref(bad), nul) == -3
    # the selection check: status word required, sizes, alignment
    assert lib.mla_check_selection(GOOD, 8, GOOD, 1, 1, 16, nul, nul) == -1
    assert lib.mla_check_selection(nul, 8, GOOD, 1, 1, 16, GOOD, nul) == -1
    assert lib.mla_check_selection(MISALIGNED, 8, GOOD, 1, 1, 16, GOOD, nul) == -2
    assert lib.mla_check_selection(GOOD, 8, GOOD, 1, 1, (1 << 20) + 1, GOOD, nul) == -3
    assert lib.mla_check_selection(GOOD, 8, GOOD, 2049, 2, 16, GOOD, nul) == -3
    assert lib.mla_check_selection(GOOD, 0, GOOD, 1, 1, 16, GOOD, nul) == -3
    assert lib.mla_check_selection(GOOD, 8, GOOD, 1, 0, 16, GOOD, nul) == -3
    # workspace too small
    need = lib.mla_sparse_decode_workspace_size(2, 64)
    assert lib.mla_sparse_decode(GOOD, GOOD, GOOD, 16, GOOD, 64, GOOD, 2, 1.0, nul, GOOD, GOOD, need - 1, nul,
                                 nul) == -4


def test_status_strings():
    assert mla.status_string(0) == "ok"
    for code in (-1, -2, -3, -4, -5, -6):
        assert mla.status_string(code) not in ("ok", "unknown status code")
    assert "end_pos" in mla.status_string(1)
    assert "timed out" in mla.status_string(4)
    assert "exchange range" in mla.status_string(8)
    assert "repeated position" in mla.status_string(16)
    # every combination of device bits names each of its bits
    for code in range(1, 32):
        s = mla.status_string(code)
        assert ("end_pos" in s) == bool(code & 1)
        assert ("rotary table" in s) == bool(code & 2)
        assert ("timed out" in s) == bool(code & 4)
        assert ("exchange range" in s) == bool(code & 8)
        assert ("repeated position" in s) == bool(code & 16)
    assert mla.status_string(-99) == "unknown status code"
    assert mla.status_string(32) == "unknown status code"


def test_python_wrappers_reject_cpu_tensors():
    import torch
    x = torch.zeros(1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mla.mla_rope_apply(x, torch.zeros(16, 32, 2), torch.ones(1, dtype=torch.int32))


def test_packed_host_inputs_are_disjoint_aligned_views():
    # the host pipeline copies a step's four inputs as one buffer: each view
    # starts on a 256-byte boundary, has its tensor's shape and touches no other
    import torch
    B, K = 5, 300
    n = mla.HostDecodeStep.packed_bytes(B, K)
    buf = torch.zeros(n, dtype=torch.uint8)
    q_nope, q_pe, topk, end = mla.HostDecodeStep.packed_inputs(buf, B, K)
    assert q_nope.shape == (B, mla.N_HEADS, mla.D_NOPE) and q_nope.dtype == torch.bfloat16
    assert q_pe.shape == (B, mla.N_HEADS, mla.D_ROPE) and q_pe.dtype == torch.bfloat16
    assert topk.shape == (B, K) and topk.dtype == torch.int32
    assert end.shape == (B,) and end.dtype == torch.int32
    base = buf.data_ptr()
    spans = []
    for t in (q_nope, q_pe, topk, end):
        off = t.data_ptr() - base
        assert off % 256 == 0
        spans.append((off, off + t.numel() * t.element_size()))
    spans.sort()
    assert spans[-1][1] <= n and all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))
    for i, t in enumerate((q_nope, q_pe, topk, end)):
        t.view(torch.uint8).fill_(i + 1)
    assert int((buf == 1).sum()) == q_nope.numel() * 2
    assert int((buf == 4).sum()) == end.numel() * 4


@pytest.mark.parametrize("B,K", [(1, 1001), (3, 256), (64, 2048), (4096, 64)])
def test_packed_host_inputs_layout(B, K):
    # the host-buffer step copies its four inputs in as one buffer: each part at a
    # 256-byte aligned offset, in order, not overlapping, with the shapes and
    # dtypes of the separate inputs
    import torch
    n = mla.HostDecodeStep.packed_bytes(B, K)
    buf = torch.zeros(n, dtype=torch.uint8)
    parts = mla.HostDecodeStep.packed_inputs(buf, B, K)
    want = [((B, 128, 128), torch.bfloat16), ((B, 128, 64), torch.bfloat16), ((B, K), torch.int32),
            ((B,), torch.int32)]
    base = buf.data_ptr()
    end = 0
    for v, (shape, dtype) in zip(parts, want):
        assert tuple(v.shape) == shape and v.dtype == dtype and v.is_contiguous()
        off = v.data_ptr() - base
        assert off % 256 == 0 and off >= end
        end = off + v.numel() * v.element_size()
    assert end <= n < end + 256
    # writing through one view leaves the others untouched
    parts[2].fill_(-1)
    assert int(parts[0].view(torch.int16).abs().sum()) == 0 and int(parts[3].sum()) == 0
