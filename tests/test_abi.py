"""The C ABI library on a machine without a GPU: it loads, exports every entry
point the header declares, and rejects bad arguments on the host before any
CUDA call is made."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build_library()
    import kda_delta_rule_fwd_gb300 as m
    return m, m.load()


def _declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(kda_\w+)\s*\(", src)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    m, L = lib
    declared = _declared_functions()
    assert {"kda_fwd", "kda_decode", "kda_workspace_size", "kda_read_device_status",
            "kda_status_string"} <= set(declared)
    for name in declared:
        assert hasattr(L, name), f"{name} declared in include/ but not exported"


def test_status_strings_and_version(lib):
    m, L = lib
    for code in range(8):
        s = m.status_string(code)
        assert s and s != "unknown status"
    assert m.status_string(99) == "unknown status"
    assert m.version().startswith("kda-gb300")


def _shape(m, **kw):
    d = dict(B=2, T=100, H=4, dk=128, dv=128, num_seqs=0, in_dtype=m.KDA_BF16,
             out_dtype=m.KDA_F32, scale=128 ** -0.5)
    d.update(kw)
    return m.Shape(**d)


def test_workspace_size(lib):
    m, L = lib
    assert L.kda_workspace_size(None) == 0
    assert m.workspace_size(_shape(m)) == 256
    # packed batches add a 64-entry-aligned int32 order list
    assert m.workspace_size(_shape(m, B=1, num_seqs=1)) == 256 + 256
    assert m.workspace_size(_shape(m, B=1, num_seqs=65)) == 256 + 512


FAKE = 1 << 32  # an aligned, never-dereferenced stand-in for a device pointer


def _fwd(L, shape, *, q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, cu=None, h0=None, out=FAKE,
         hT=None, ws=FAKE, ws_bytes=1 << 20):
    vp = ctypes.c_void_p
    return L.kda_fwd(None if shape is None else ctypes.byref(shape), vp(q), vp(k), vp(v), vp(g),
                     vp(beta), vp(cu), vp(h0), vp(out), vp(hT), vp(ws), ws_bytes, None)


def _decode(L, shape, *, state=FAKE, out=FAKE, ws=FAKE, ws_bytes=1 << 20, beta=FAKE):
    vp = ctypes.c_void_p
    return L.kda_decode(ctypes.byref(shape), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(beta),
                        vp(state), vp(out), vp(ws), ws_bytes, None)


def test_argument_errors_return_before_launch(lib):
    m, L = lib
    assert _fwd(L, None) == m.KDA_ERR_INVALID_ARG
    assert _fwd(L, _shape(m, H=0)) == m.KDA_ERR_INVALID_ARG
    assert _fwd(L, _shape(m, T=-1)) == m.KDA_ERR_INVALID_ARG
    assert _fwd(L, _shape(m, in_dtype=7)) == m.KDA_ERR_INVALID_ARG
    assert _fwd(L, _shape(m, scale=float("nan"))) == m.KDA_ERR_INVALID_ARG
    assert _fwd(L, _shape(m, dk=96, dv=96)) == m.KDA_ERR_UNSUPPORTED
    assert _fwd(L, _shape(m, dk=128, dv=64)) == m.KDA_ERR_UNSUPPORTED
    assert _fwd(L, _shape(m), q=0) == m.KDA_ERR_INVALID_ARG
    assert _fwd(L, _shape(m), out=0) == m.KDA_ERR_INVALID_ARG
    assert _fwd(L, _shape(m), k=FAKE + 8) == m.KDA_ERR_INVALID_ARG       # not 16-byte aligned
    assert _fwd(L, _shape(m), h0=FAKE + 4) == m.KDA_ERR_INVALID_ARG
    assert _fwd(L, _shape(m), beta=FAKE + 1) == m.KDA_ERR_INVALID_ARG    # bf16 beta misaligned
    assert _fwd(L, _shape(m), ws=0) == m.KDA_ERR_WORKSPACE
    assert _fwd(L, _shape(m), ws=FAKE + 16) == m.KDA_ERR_WORKSPACE       # not 256-byte aligned
    assert _fwd(L, _shape(m), ws_bytes=255) == m.KDA_ERR_WORKSPACE
    # packed batches need B == 1 and room for the order list
    assert _fwd(L, _shape(m, B=2, num_seqs=3), cu=FAKE) == m.KDA_ERR_INVALID_ARG
    assert _fwd(L, _shape(m, B=1, num_seqs=3), cu=FAKE, ws_bytes=256) == m.KDA_ERR_WORKSPACE
    assert _fwd(L, _shape(m, B=1, num_seqs=3), cu=FAKE + 2) == m.KDA_ERR_INVALID_ARG
    # decode: 1..8 tokens per step
    assert _decode(L, _shape(m, T=0)) == m.KDA_ERR_UNSUPPORTED
    assert _decode(L, _shape(m, T=9)) == m.KDA_ERR_UNSUPPORTED
    assert _decode(L, _shape(m, T=1), state=0) == m.KDA_ERR_INVALID_ARG
    assert _decode(L, _shape(m, T=1), state=FAKE + 8) == m.KDA_ERR_INVALID_ARG
    assert _decode(L, _shape(m, T=1), ws_bytes=0) == m.KDA_ERR_WORKSPACE


def _decode_commit(L, shape, *, counts=FAKE, out=FAKE, state=FAKE, ws_bytes=1 << 20):
    vp = ctypes.c_void_p
    return L.kda_decode_commit(ctypes.byref(shape), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                               vp(FAKE), vp(counts), vp(state), vp(out), vp(FAKE), ws_bytes, None)


def test_decode_commit_argument_errors(lib):
    """Commit counts are required; outputs are optional only here; the counts must
    be 4-byte aligned; the step-size and workspace rules are kda_decode's."""
    m, L = lib
    L.kda_decode_commit.restype = ctypes.c_int
    assert _decode_commit(L, _shape(m, T=4), counts=0) == m.KDA_ERR_INVALID_ARG
    assert _decode_commit(L, _shape(m, T=4), counts=FAKE + 2) == m.KDA_ERR_INVALID_ARG
    assert _decode_commit(L, _shape(m, T=9)) == m.KDA_ERR_UNSUPPORTED
    assert _decode_commit(L, _shape(m, T=4), state=0) == m.KDA_ERR_INVALID_ARG
    assert _decode_commit(L, _shape(m, T=4), ws_bytes=0) == m.KDA_ERR_WORKSPACE
    assert _decode(L, _shape(m, T=4), out=0) == m.KDA_ERR_INVALID_ARG  # kda_decode needs out
    if not torch.cuda.is_available():  # valid arguments reach the (absent) device
        assert _decode_commit(L, _shape(m, T=4), out=0) == m.KDA_ERR_CUDA


def _fwd_ckpt(L, shape, *, interval=512, ckpt=FAKE, offs=None, rows=8, cu=None):
    vp = ctypes.c_void_p
    L.kda_fwd_checkpoints.restype = ctypes.c_int
    return L.kda_fwd_checkpoints(ctypes.byref(shape), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                                 vp(FAKE), vp(cu), vp(None), vp(FAKE), vp(FAKE),
                                 ctypes.c_int32(interval), vp(ckpt), vp(offs),
                                 ctypes.c_int64(rows), vp(FAKE), ctypes.c_size_t(1 << 20), None)


def test_fwd_checkpoints_argument_errors(lib):
    """The interval is a positive multiple of the chunk length; the buffer is
    required and aligned; packed batches need row offsets."""
    m, L = lib
    for bad in (0, -64, 100, 32):
        assert _fwd_ckpt(L, _shape(m), interval=bad) == m.KDA_ERR_INVALID_ARG
    assert _fwd_ckpt(L, _shape(m), ckpt=0) == m.KDA_ERR_INVALID_ARG
    assert _fwd_ckpt(L, _shape(m), ckpt=FAKE + 4) == m.KDA_ERR_INVALID_ARG
    assert _fwd_ckpt(L, _shape(m), rows=-1) == m.KDA_ERR_INVALID_ARG
    packed = _shape(m, B=1, num_seqs=3)
    assert _fwd_ckpt(L, packed, cu=FAKE) == m.KDA_ERR_INVALID_ARG             # no offsets
    assert _fwd_ckpt(L, packed, cu=FAKE, offs=FAKE + 2) == m.KDA_ERR_INVALID_ARG
    assert _fwd_ckpt(L, _shape(m, dk=96, dv=96)) == m.KDA_ERR_UNSUPPORTED   # kda_fwd's rules
    if not torch.cuda.is_available():  # valid arguments reach the (absent) device
        assert _fwd_ckpt(L, _shape(m)) == m.KDA_ERR_CUDA
        assert _fwd_ckpt(L, packed, cu=FAKE, offs=FAKE) == m.KDA_ERR_CUDA


@pytest.mark.skipif(torch.cuda.is_available(), reason="would launch on fake pointers")
def test_valid_call_without_a_gpu_reports_cuda_error(lib):
    """With valid arguments the first CUDA call fails on a GPU-less host, and the
    library maps that to KDA_ERR_CUDA instead of crashing."""
    m, L = lib
    assert _fwd(L, _shape(m)) == m.KDA_ERR_CUDA
    assert _decode(L, _shape(m, T=8)) == m.KDA_ERR_CUDA
    assert L.kda_read_device_status(ctypes.c_void_p(FAKE), None) == m.KDA_ERR_CUDA
    assert L.kda_read_device_status(ctypes.c_void_p(FAKE + 16), None) == m.KDA_ERR_WORKSPACE


def test_binding_refuses_to_run_without_library(tmp_path):
    import kda_delta_rule_fwd_gb300 as m
    with pytest.raises(RuntimeError, match="not built"):
        m.load(str(tmp_path / "missing.so"))


def test_workspace_size_long_chain_split(lib):
    """A fixed-length bf16 batch of few, very long chains reserves (3 nseg - 2)
    segment states of 128x128 fp32 per chain.  The plan minimises the finishing time
    of the items on 152 SMs, each SM taking the next item when free: a chain's first
    launch runs segment 0 from its start state (all chains' first) beside 2 (nseg - 2)
    transition items, the second the other nseg - 1 segments, and segment 0 may be up
    to 3 times as long as the others.  B=1, T=2^20, H=32 (16384 chunks) -> 5 segments,
    segment 0 of 5460 chunks and the others of 2731: the 32 long items and 120 short
    ones start together, the other 72 short ones follow on the 120 SMs, so the first
    launch ends at 5462 and the second (128 items) at 2731 more: 8195.5 chunk-steps
    with the scan, against 9833.5 for 5 equal segments; B=1, T=64*255, H=2 -> 3."""
    m, L = lib
    assert m.workspace_size(_shape(m, B=1, T=1 << 20, H=32)) == 256 + 32 * 13 * 128 * 128 * 4
    assert m.workspace_size(_shape(m, B=1, T=64 * 255, H=2)) == 256 + 2 * 7 * 128 * 128 * 4
    # one chain: every split is two single waves, so more segments always model
    # faster and the cap of 64 applies (190 states)
    assert m.workspace_size(_shape(m, B=1, T=1 << 20, H=1)) == 256 + 190 * 128 * 128 * 4
    # 8 chains of 1024 chunks: 11 segments of 94 chunks take 1 + 1 waves (152 and 80
    # items; 188 chunk-steps + 5.5 of scan); 16 segments of 64 chunks take 2 + 1
    # (192 + 8), 10 of 103 chunks 1 + 1 (206 + 5)
    assert m.workspace_size(_shape(m, B=8, T=1 << 16, H=1)) == 256 + 8 * 31 * 128 * 128 * 4
    # 64 chains: 3 segments, segment 0 of 8192 chunks beside the 128 transition items
    # of segment 1 (4096 chunks each, on the other 88 SMs and then 40 of them), then
    # 128 output items: 12289.5 chunk-steps against 16384 for the chains whole
    assert m.workspace_size(_shape(m, B=2, T=1 << 20, H=32)) == 256 + 64 * 7 * 128 * 128 * 4
    # float32 inputs, many chains or short chains never split
    assert m.workspace_size(_shape(m, B=1, T=1 << 20, H=32, in_dtype=m.KDA_F32)) == 256
    assert m.workspace_size(_shape(m, B=4, T=4096, H=32)) == 256
    assert m.workspace_size(_shape(m, B=1, T=64 * 127, H=2)) == 256
    # the split is optional: the minimum workspace is still accepted
    if not torch.cuda.is_available():  # would launch on fake pointers otherwise
        assert _fwd(L, _shape(m, B=1, T=1 << 20, H=32), ws_bytes=256) == m.KDA_ERR_CUDA


def _fwd_pre(L, m, shape, pre, *, g=FAKE):
    vp = ctypes.c_void_p
    L.kda_fwd_preproc.restype = ctypes.c_int
    return L.kda_fwd_preproc(ctypes.byref(shape), ctypes.byref(pre) if pre else None, vp(FAKE),
                             vp(FAKE), vp(FAKE), vp(g), vp(FAKE), None, None, vp(FAKE),
                             vp(FAKE), vp(FAKE), ctypes.c_size_t(1 << 20), None)


def _dec_pre(L, m, shape, pre, *, g=FAKE):
    vp = ctypes.c_void_p
    L.kda_decode_preproc.restype = ctypes.c_int
    return L.kda_decode_preproc(ctypes.byref(shape), ctypes.byref(pre) if pre else None,
                                vp(FAKE), vp(FAKE), vp(FAKE), vp(g), vp(FAKE), vp(FAKE),
                                vp(FAKE), vp(FAKE), ctypes.c_size_t(1 << 20), None)


def test_preproc_argument_errors(lib):
    """A per-head gate scale needs the softplus step and 4-byte alignment; a
    per-channel g needs 16-byte alignment, a per-head g only its dtype's."""
    m, L = lib
    P = m.Preproc
    for call, shp in ((_fwd_pre, _shape(m)), (_dec_pre, _shape(m, T=2))):
        assert call(L, m, shp, P(1, 0, 1, 0, FAKE)) == m.KDA_ERR_INVALID_ARG  # scale, no softplus
        assert call(L, m, shp, P(1, 1, 1, 0, FAKE + 2)) == m.KDA_ERR_INVALID_ARG
        assert call(L, m, shp, P(0, 1, 0, 0, None), g=FAKE + 2) == m.KDA_ERR_INVALID_ARG
        assert call(L, m, shp, None, g=FAKE + 2) == m.KDA_ERR_INVALID_ARG
        assert call(L, m, shp, P(0, 1, 0, 1, None), g=FAKE + 1) == m.KDA_ERR_INVALID_ARG
        if not torch.cuda.is_available():  # valid arguments reach the (absent) device
            assert call(L, m, shp, P(0, 1, 0, 1, FAKE), g=FAKE + 2) == m.KDA_ERR_CUDA
            assert call(L, m, shp, P(1, 1, 1, 0, FAKE + 4)) == m.KDA_ERR_CUDA


def _bwd(L, shape, *, dout=FAKE, dq=FAKE, dbeta=FAKE, dh0=None, ws_bytes=None, cu=None):
    vp = ctypes.c_void_p
    L.kda_bwd.restype = ctypes.c_int
    L.kda_bwd_workspace_size.restype = ctypes.c_size_t
    L.kda_bwd_workspace_size.argtypes = [ctypes.c_void_p]
    if ws_bytes is None:
        ws_bytes = L.kda_bwd_workspace_size(ctypes.byref(shape))
    return L.kda_bwd(ctypes.byref(shape), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                     vp(cu), None, vp(dout), None, vp(dq), vp(FAKE), vp(FAKE), vp(FAKE),
                     vp(dbeta), vp(dh0), vp(FAKE), ctypes.c_size_t(ws_bytes), None)


def test_bwd_workspace_and_argument_errors(lib):
    """The backward keeps, per 16-token sub-chunk and head, the float32 start state
    (dk x dv) with the sub-chunk's X and U (16 x dv) and T and P (16 x 16): the
    workspace size says so, and a smaller workspace, a missing or misaligned
    gradient buffer or an unsupported head size is refused before any launch."""
    m, L = lib
    shp = _shape(m, B=2, T=100, H=4)
    L.kda_bwd_workspace_size.restype = ctypes.c_size_t
    L.kda_bwd_workspace_size.argtypes = [ctypes.c_void_p]
    need = L.kda_bwd_workspace_size(ctypes.byref(shp))
    row = (128 * 128 + 2 * 16 * 128 + 2 * 16 * 16) * 4
    assert need >= 2 * 7 * 4 * row                     # ceil(100 / 16) = 7 sub-chunks
    assert need < 2 * 7 * 4 * row + 4096
    packed = _shape(m, B=1, T=100, H=4, num_seqs=3)
    assert L.kda_bwd_workspace_size(ctypes.byref(packed)) >= (7 + 3) * 4 * row
    assert _bwd(L, shp, ws_bytes=need - 1) == m.KDA_ERR_WORKSPACE
    assert _bwd(L, shp, dout=0) == m.KDA_ERR_INVALID_ARG
    assert _bwd(L, shp, dq=0) == m.KDA_ERR_INVALID_ARG
    assert _bwd(L, shp, dq=FAKE + 4) == m.KDA_ERR_INVALID_ARG
    assert _bwd(L, shp, dbeta=FAKE + 2) == m.KDA_ERR_INVALID_ARG
    assert _bwd(L, shp, dh0=FAKE + 8) == m.KDA_ERR_INVALID_ARG
    assert _bwd(L, _shape(m, dk=96, dv=96)) == m.KDA_ERR_UNSUPPORTED
    assert _bwd(L, packed, cu=FAKE + 2) == m.KDA_ERR_INVALID_ARG
    if not torch.cuda.is_available():  # valid arguments reach the (absent) device
        assert _bwd(L, shp) == m.KDA_ERR_CUDA
        assert _bwd(L, packed, cu=FAKE) == m.KDA_ERR_CUDA


def test_workspace_size_packed_long_chain_split(lib):
    """A packed bf16 batch of at least 2 * 64 chunks may hold a sequence the device
    planner splits: the workspace then reserves the plan (header, four int32 per
    sequence, the item tables) and 3 * ns_max float32 states per head, ns_max =
    T / 4096 + T / 524288 + 2 bounding the split sequences' segments."""
    m, L = lib
    assert m.workspace_size(_shape(m, B=1, T=8191, H=32, num_seqs=4)) == 256 + 256
    T, H, N = 267445, 2, 4
    ns = T // 4096 + T // 524288 + 2
    plan = 16 + N * 16 + ns * 8 + ns * 4 + (N + ns) * 8
    plan = (plan + 255) // 256 * 256
    assert m.workspace_size(_shape(m, B=1, T=T, H=H, num_seqs=N)) == \
        256 + 256 + plan + 3 * ns * H * 128 * 128 * 4
    # float32 inputs run the float32 kernel, which never splits
    assert m.workspace_size(_shape(m, B=1, T=T, H=H, num_seqs=N, in_dtype=m.KDA_F32)) == 512
