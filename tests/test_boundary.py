"""Host-only checks of the C ABI (no GPU needed, nothing is launched).

Every falcon_fwd call below is invalid by construction, so the library must
return its error code from the synchronous argument check before any launch.
"""

import ctypes
import os
import re

import pytest

from weight_linear_attention_gb300 import build as fbuild
from weight_linear_attention_gb300 import falcon as F

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return F.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "falcon.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\*\s]+?\b(falcon_\w+)\s*\(", src, flags=re.M)))


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert set(names) == set(F.EXPORTED), names
    for n in names:
        assert hasattr(lib, n), n
    assert F.falcon_abi_version() == 4


def test_dims_struct_layout():
    assert ctypes.sizeof(F.FalconDims) == 64
    assert F.FalconDims.pos.offset == 48 and F.FalconDims.eps.offset == 56


def test_status_strings(lib):
    for s in range(6):
        assert F.status_string(s)
    assert F.status_string(99) == "unknown status"


def test_tail_bytes(lib):
    d = F.make_dims(2, 3, 100, 64, 32, window=4, dtype=F.FALCON_BF16)
    assert F.falcon_tail_bytes(d) == 2 * 3 * (4 * 64 + 3 * 32) * 2
    d = F.make_dims(2, 3, 100, 64, 32, window=1, dtype=F.FALCON_F32)
    assert F.falcon_tail_bytes(d) == 2 * 3 * 64 * 4


@pytest.mark.parametrize("case,expect", [
    (dict(), 1),
    (dict(dtype=F.FALCON_F32, dk=16, dv=16, chunk=16), 1),
    (dict(variant=F.FALCON_3, window=4, chunk=32), 1),
    (dict(variant=F.FALCON_2A), 1),                 # inner-product variants: CUDA-core kernel
    (dict(variant=F.FALCON_3A, window=3, chunk=32), 1),
    (dict(variant=F.FALCON_3A, window=4, chunk=64), 0),  # chunk*window > 128
    (dict(variant=7), 0),
    (dict(window=2), 0),                            # window only for Falcon-3
    (dict(variant=F.FALCON_3, window=9, chunk=16), 0),
    (dict(variant=F.FALCON_3, window=4, chunk=64), 0),  # chunk*window > 128
    (dict(dk=48), 0),
    (dict(dv=256), 0),
    (dict(chunk=128), 0),
    (dict(chunk=0), 0),
    (dict(dtype=7), 0),
    (dict(eps_gamma=0.0), 0),
    (dict(eps_gamma=1.0), 0),
    (dict(eps=-1.0), 0),
    (dict(seqlen=-1), 0),
])
def test_kernel_for_validation(lib, case, expect):
    c = dict(variant=F.FALCON_1, batch=8, heads=12, seqlen=1024, dk=64, dv=64, window=1, dtype=F.FALCON_BF16,
             chunk=64)
    c.update(case)
    d = F.make_dims(c["batch"], c["heads"], c["seqlen"], c["dk"], c["dv"], window=c["window"], dtype=c["dtype"],
                    eps=c.get("eps", 1e-6), eps_gamma=c.get("eps_gamma", 1e-6))
    got = F.falcon_kernel_for(c["variant"], d, c["chunk"])
    assert (got != 0) == bool(expect), (case, got)


# Fake device addresses: never dereferenced because every call below is rejected.
A = 1 << 40


def _call(variant=F.FALCON_1, q=A, k=A + (1 << 30), v=A + (2 << 30), beta=A + (3 << 30), lam=A + (4 << 30),
          S0=None, tail=None, out=A + (5 << 30), S_final=None, tail_out=None, dims=None, chunk=64, ws=None,
          ws_bytes=0):
    if dims is None:
        dims = F.make_dims(2, 2, 64, 64, 64)
    return F.falcon_fwd(variant, q, k, v, beta, lam, S0, tail, out, S_final, tail_out, dims, chunk, ws, ws_bytes,
                        stream=0)


def test_null_required_pointers(lib):
    for name in ("q", "k", "v", "beta", "lam", "out"):
        assert _call(**{name: 0}) == F.FALCON_ERR_INVALID_ARG, name


def test_misaligned_pointers(lib):
    assert _call(q=A + 2) == F.FALCON_ERR_MISALIGNED
    assert _call(out=A + (5 << 30) + 8) == F.FALCON_ERR_MISALIGNED
    assert _call(S0=A + (6 << 30) + 4) == F.FALCON_ERR_MISALIGNED
    assert _call(beta=A + (3 << 30) + 2) == F.FALCON_ERR_MISALIGNED


def test_tail_and_pos_must_agree(lib):
    d = F.make_dims(2, 2, 64, 64, 64, pos=10)
    assert _call(dims=d) == F.FALCON_ERR_INVALID_ARG               # pos > 0 without a tail
    assert _call(tail=A + (7 << 30)) == F.FALCON_ERR_INVALID_ARG   # tail with pos == 0


def test_out_must_not_overlap_inputs(lib):
    assert _call(out=A + 4096) == F.FALCON_ERR_INVALID_ARG          # inside q
    assert _call(out=A + (2 << 30) - 4096) == F.FALCON_ERR_INVALID_ARG  # runs into v
    assert _call(S0=A + (5 << 30), S_final=A + (8 << 30)) == F.FALCON_ERR_INVALID_ARG  # S0 inside out


def test_tail_out_must_not_overlap_tail(lib):
    d = F.make_dims(2, 2, 64, 64, 64, pos=10, eps_gamma=2.0)        # also invalid eps_gamma: never launches
    assert _call(dims=d, tail=A + (7 << 30), tail_out=A + (7 << 30)) == F.FALCON_ERR_INVALID_ARG


def test_unsupported_and_invalid_shapes(lib):
    assert _call(dims=F.make_dims(2, 2, 64, 48, 64)) == F.FALCON_ERR_UNSUPPORTED
    assert _call(variant=8) == F.FALCON_ERR_INVALID_ARG
    assert _call(variant=0) == F.FALCON_ERR_INVALID_ARG
    assert _call(chunk=-4) == F.FALCON_ERR_INVALID_ARG
    assert _call(chunk=24) == F.FALCON_ERR_UNSUPPORTED
    assert _call(dims=F.make_dims(2, 2, 64, 64, 64, window=3)) == F.FALCON_ERR_INVALID_ARG


@pytest.mark.parametrize("case,expect", [
    (dict(), 6),                                           # Falcon-1, bf16, 64, chunk 64: fused kernel
    (dict(variant=F.FALCON_1A), 6),
    (dict(variant=F.FALCON_1, seqlen=0), 6),          # no tokens: the fused kernel still writes S_final, tail
    (dict(chunk=32), 1),
    (dict(dtype=F.FALCON_F32), 1),
    (dict(variant=F.FALCON_2), 7),                        # Falcon-2 / 2A, bf16, 64, chunk 64: per-column kernel
    (dict(variant=F.FALCON_2, dtype=F.FALCON_F32), 1),
    (dict(variant=F.FALCON_2, chunk=32), 1),
    (dict(dk=32, dv=32), 1),
    (dict(seqlen=1), 4),                                  # one token: the single-token kernel
    (dict(seqlen=1, variant=F.FALCON_1A, dtype=F.FALCON_F32), 4),
    (dict(seqlen=1, variant=F.FALCON_2), 4),
    (dict(seqlen=1, dk=32, dv=32), 1),
    (dict(seqlen=2), 6),
    (dict(variant=F.FALCON_2A), 7),
    (dict(variant=F.FALCON_2A, seqlen=0), 7),
    (dict(variant=F.FALCON_2A, seqlen=1), 4),            # ... and the single-token kernel for 2A
])
def test_kernel_choice(lib, case, expect):
    c = dict(variant=F.FALCON_1, seqlen=1024, dk=64, dv=64, dtype=F.FALCON_BF16, chunk=64)
    c.update(case)
    d = F.make_dims(8, 12, c["seqlen"], c["dk"], c["dv"], dtype=c["dtype"])
    assert F.falcon_kernel_for(c["variant"], d, c["chunk"]) == expect


def test_workspace_bytes(lib):
    # the fused kernel (Falcon-1 / 1A, bf16, 64, chunk 64) keeps everything on chip: no workspace
    assert F.falcon_workspace_bytes(F.FALCON_1, F.make_dims(8, 12, 1024, 64, 64), 64) == 0
    assert F.falcon_workspace_bytes(F.FALCON_1A, F.make_dims(2, 3, 65, 64, 64), 64) == 0
    assert F.falcon_workspace_bytes(F.FALCON_1, F.make_dims(2, 3, 0, 64, 64), 64) == 0
    assert F.falcon_workspace_bytes(F.FALCON_2, F.make_dims(2, 3, 64, 64, 64), 64) == 0
    assert F.falcon_workspace_bytes(F.FALCON_1, F.make_dims(2, 3, 64, 64, 64, dtype=F.FALCON_F32), 64) == 0
    assert F.falcon_workspace_bytes(F.FALCON_1, F.make_dims(2, 3, 64, 64, 64), 32) == 0
    assert F.falcon_workspace_bytes(F.FALCON_2A, F.make_dims(2, 3, 64, 64, 64), 64) == 0
    assert F.falcon_workspace_bytes(F.FALCON_1, F.make_dims(8, 12, 1, 64, 64), 64) == 0  # single-token kernel


def test_workspace_checks(lib):
    # Falcon-1 at chunk 32 over 4 sequences of 256 tokens: the scan path, which uses a workspace
    d = F.make_dims(2, 2, 256, 64, 64)
    need = F.falcon_workspace_bytes(F.FALCON_1, d, 32)
    assert need > 0
    W = A + (9 << 30)
    assert _call(dims=d, chunk=32, ws=W, ws_bytes=need - 1) == F.FALCON_ERR_INVALID_ARG      # too small
    assert _call(dims=d, chunk=32, ws=W + 128, ws_bytes=need) == F.FALCON_ERR_MISALIGNED    # 256-byte alignment
    assert _call(dims=d, chunk=32, ws=A + 4096, ws_bytes=need) == F.FALCON_ERR_INVALID_ARG   # overlaps q
    assert _call(dims=d, chunk=32, ws=A + (5 << 30) - 4096, ws_bytes=need) == F.FALCON_ERR_INVALID_ARG  # runs into out
    # a well-formed workspace with an otherwise invalid call is still rejected before any launch
    assert _call(dims=d, chunk=24, ws=W, ws_bytes=need) == F.FALCON_ERR_UNSUPPORTED


def test_written_buffers_must_not_overlap_anything(lib):
    # S_final and tail_out, like out, may overlap no input and no other written buffer (S_final may
    # only equal S0 exactly: an in-place state update)
    d = F.make_dims(2, 2, 64, 64, 64, pos=3)
    tl = A + (7 << 30)
    assert _call(S_final=A + 4096) == F.FALCON_ERR_INVALID_ARG                       # inside q
    assert _call(S_final=A + (4 << 30)) == F.FALCON_ERR_INVALID_ARG                  # on lambda
    assert _call(S_final=A + (5 << 30) + 256) == F.FALCON_ERR_INVALID_ARG            # inside out
    assert _call(S0=A + (6 << 30), S_final=A + (6 << 30) + 64) == F.FALCON_ERR_INVALID_ARG  # shifted onto S0
    assert _call(dims=d, tail=tl, tail_out=A + (1 << 30)) == F.FALCON_ERR_INVALID_ARG  # on k
    assert _call(dims=d, tail=tl, tail_out=A + (5 << 30)) == F.FALCON_ERR_INVALID_ARG  # on out
    assert _call(dims=d, tail=tl, S_final=A + (8 << 30), tail_out=A + (8 << 30) + 512) == F.FALCON_ERR_INVALID_ARG
    assert _call(dims=d, tail=tl, S0=A + (8 << 30), tail_out=A + (8 << 30)) == F.FALCON_ERR_INVALID_ARG  # on S0


def test_binding_raises_when_library_missing(tmp_path):
    with pytest.raises(RuntimeError):
        F.load(str(tmp_path / "nope.so"))


# ---------------------------------------------------------------- falcon_bwd (host-side checks only)

def _bwd(variant=F.FALCON_1, dims=None, chunk=64, ws=A + (20 << 30), ws_bytes=None, **kw):
    if dims is None:
        dims = F.make_dims(2, 2, 64, 64, 64)
    if ws_bytes is None:
        ws_bytes = F.falcon_bwd_workspace_bytes(F.FALCON_1, dims, 64)
    p = dict(q=A, k=A + (1 << 30), v=A + (2 << 30), beta=A + (3 << 30), lam=A + (4 << 30), S0=None, tail=None,
             dout=A + (5 << 30), dS_final=None, dq=A + (10 << 30), dk=A + (11 << 30), dv=A + (12 << 30),
             dbeta=A + (13 << 30), dlam=A + (14 << 30), dS0=None, dtail=None)
    p.update(kw)
    return F.falcon_bwd(variant, p["q"], p["k"], p["v"], p["beta"], p["lam"], p["S0"], p["tail"], p["dout"],
                        p["dS_final"], p["dq"], p["dk"], p["dv"], p["dbeta"], p["dlam"], p["dS0"], p["dtail"], dims,
                        chunk, ws, ws_bytes, stream=0)


def test_bwd_workspace_bytes(lib):
    # B*H*ceil(T/64) chunks of six 64 x 64 x 4-byte slots (U and V in fp32; M, T, S_n and dS_{n+1}
    # each as bf16 hi and lo tiles) and 3 KiB of the chunk's scalars
    assert F.falcon_bwd_workspace_bytes(F.FALCON_1, F.make_dims(8, 12, 1024, 64, 64), 64) == 8 * 12 * 16 * 101376
    assert F.falcon_bwd_workspace_bytes(F.FALCON_1A, F.make_dims(2, 3, 65, 64, 64, dtype=F.FALCON_F32), 64) \
        == 2 * 3 * 2 * 101376
    assert F.falcon_bwd_workspace_bytes(F.FALCON_1, F.make_dims(2, 3, 0, 64, 64), 64) == 0
    for v in (F.FALCON_2, F.FALCON_2A, F.FALCON_3, F.FALCON_3A):  # no backward kernel for these yet
        assert F.falcon_bwd_workspace_bytes(v, F.make_dims(2, 3, 64, 64, 64, window=2 if v >= 5 else 1), 64) == 0
    assert F.falcon_bwd_workspace_bytes(F.FALCON_1, F.make_dims(2, 3, 64, 32, 32), 64) == 0
    assert F.falcon_bwd_workspace_bytes(F.FALCON_1, F.make_dims(2, 3, 64, 64, 64), 32) == 0


def test_bwd_argument_checks(lib):
    assert _bwd(variant=F.FALCON_2) == F.FALCON_ERR_UNSUPPORTED
    assert _bwd(chunk=32) == F.FALCON_ERR_UNSUPPORTED
    assert _bwd(dims=F.make_dims(2, 2, 64, 32, 32)) == F.FALCON_ERR_UNSUPPORTED
    for name in ("q", "dout", "dq", "dk", "dv", "dbeta", "dlam"):
        assert _bwd(**{name: 0}) == F.FALCON_ERR_INVALID_ARG, name
    assert _bwd(ws=None, ws_bytes=0) == F.FALCON_ERR_INVALID_ARG              # the workspace is required
    assert _bwd(ws_bytes=1000) == F.FALCON_ERR_INVALID_ARG                    # too small
    assert _bwd(ws=A + (20 << 30) + 128) == F.FALCON_ERR_MISALIGNED
    assert _bwd(dq=A + (10 << 30) + 4) == F.FALCON_ERR_MISALIGNED
    assert _bwd(dbeta=A + (13 << 30) + 2) == F.FALCON_ERR_MISALIGNED
    assert _bwd(dq=A + 1024) == F.FALCON_ERR_INVALID_ARG                      # a gradient over an input
    assert _bwd(dk=A + (10 << 30) + 4096) == F.FALCON_ERR_INVALID_ARG         # two gradients overlap
    assert _bwd(ws=A + (14 << 30)) == F.FALCON_ERR_INVALID_ARG                # workspace over a gradient
    assert _bwd(dtail=A + (15 << 30)) == F.FALCON_ERR_INVALID_ARG             # dtail with pos == 0
    d = F.make_dims(2, 2, 64, 64, 64, pos=5)
    assert _bwd(dims=d) == F.FALCON_ERR_INVALID_ARG                            # pos > 0 without a tail


def test_scan_path_choice(lib):
    # Falcon-3 (W = 4) at 2 x 12 heads, 8192 tokens, chunk 32: few sequences, many chunks -> scan path,
    # workspace B*H*(N + ceil(N/16)) blocks of five 64 x 64 fp32 matrices, plus (Falcon-3) one fp32
    # window normaliser per token
    d = F.make_dims(2, 12, 8192, 64, 64, window=4)
    assert F.falcon_kernel_for(F.FALCON_3, d, 32) == 5
    assert F.falcon_workspace_bytes(F.FALCON_3, d, 32) == 24 * (256 + 16) * 5 * 64 * 64 * 4 + 24 * 8192 * 4
    assert F.falcon_workspace_bytes(F.FALCON_3A, d, 32) == 24 * (256 + 16) * 5 * 64 * 64 * 4
    assert F.falcon_kernel_for(F.FALCON_3A, d, 32) == 5
    assert F.falcon_kernel_for(F.FALCON_2, F.make_dims(2, 12, 8192, 64, 64), 64) == 7  # per-column kernel
    assert F.falcon_kernel_for(F.FALCON_2, F.make_dims(2, 12, 8192, 64, 64), 32) == 1  # per-column maps: no scan
    assert F.falcon_kernel_for(F.FALCON_3, F.make_dims(8, 12, 8192, 64, 64, window=4), 32) == 1  # many sequences
    assert F.falcon_kernel_for(F.FALCON_3, F.make_dims(2, 12, 64, 64, 64, window=4), 32) == 1  # two chunks
    assert F.falcon_kernel_for(F.FALCON_1, F.make_dims(2, 12, 8192, 64, 64), 64) == 6  # bf16 chunk 64: fused
    assert F.falcon_kernel_for(F.FALCON_1, F.make_dims(2, 12, 8192, 64, 64), 32) == 5
