"""The C-ABI library without a GPU: it loads, exports what include/gdr.h
declares, and rejects bad arguments before touching the device.

Only calls whose arguments fail validation are made here; they return before
any CUDA runtime call, so no kernel is launched.
"""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import gated_delta_rule_10_gb300 as gdr
from gated_delta_rule_10_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdr.h")


@pytest.fixture(scope="module")
def L():
    from gated_delta_rule_10_gb300 import build
    build.build()
    return gdr.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdr_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("gdr_chunk_fwd", "gdr_chunk_fwd_workspace", "gdr_recurrent_step",
              "gdr_gate_cumsum", "gdr_status_string", "gdr_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", _binding.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(L, name) is not None


def test_header_compiles_as_c_and_cpp(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "gdr.h"\nint f(void){ gdr_shape s; (void)s; return GDR_OK; }\n')
    for compiler in ("gcc", "g++"):
        subprocess.run([compiler, "-fsyntax-only", "-Wall", "-Werror", "-I",
                        os.path.join(ROOT, "include"), "-x", "c" if compiler == "gcc" else "c++",
                        str(src)], check=True)


def test_version_and_status_strings(L):
    assert L.gdr_abi_version() >= 1
    for code, name in _binding.STATUS.items():
        assert gdr.status_string(code).startswith(name)
    assert "unknown" in gdr.status_string(99)


def _shape(**kw):
    d = dict(B=1, T=64, H=1, dk=64, dv=64, dtype=_binding.GDR_BF16, flags=0, scale=0.125)
    d.update(kw)
    return _binding.Shape(**d)


def test_workspace_query(L):
    n = ctypes.c_size_t(123)
    assert L.gdr_chunk_fwd_workspace(ctypes.byref(_shape()), ctypes.byref(n)) == 0
    # bf16: status words + one packet per chunk: Q_gamma, -Y, K_tail (64 x d_k bf16 each),
    # A_qk (64 x 64 bf16), gamma_C (1 KB), U (64 x d_v bf16)
    assert n.value == 256 + 3 * 64 * 64 * 2 + 8192 + 1024 + 64 * 64 * 2
    s = _shape(B=2, T=130, H=3, dk=128, dv=128)
    assert L.gdr_chunk_fwd_workspace(ctypes.byref(s), ctypes.byref(n)) == 0
    assert n.value == 256 + 2 * 3 * 3 * 74752
    assert L.gdr_chunk_fwd_workspace_min(ctypes.byref(s), ctypes.byref(n)) == 0
    assert n.value == 256                      # the single-kernel path: status words only
    assert L.gdr_chunk_fwd_workspace_min(ctypes.byref(_shape(dtype=_binding.GDR_F32)),
                                         ctypes.byref(n)) == 0
    assert n.value == 0
    assert L.gdr_chunk_fwd_workspace_min(ctypes.byref(_shape(dk=96)), ctypes.byref(n)) == 2
    assert L.gdr_chunk_fwd_workspace(ctypes.byref(_shape(dtype=_binding.GDR_F32)),
                                     ctypes.byref(n)) == 0
    assert n.value == 0
    assert L.gdr_chunk_fwd_workspace(None, ctypes.byref(n)) == 1
    assert L.gdr_chunk_fwd_workspace(ctypes.byref(_shape()), None) == 1
    assert L.gdr_chunk_fwd_workspace(ctypes.byref(_shape(dk=96)), ctypes.byref(n)) == 2
    assert L.gdr_chunk_fwd_workspace(ctypes.byref(_shape(T=0)), ctypes.byref(n)) == 1
    assert L.gdr_chunk_fwd_workspace(ctypes.byref(_shape(flags=32)), ctypes.byref(n)) == 1
    assert L.gdr_chunk_fwd_workspace(ctypes.byref(_shape(dtype=7)), ctypes.byref(n)) == 1
    assert L.gdr_chunk_fwd_workspace(ctypes.byref(_shape(scale=float("nan"))),
                                     ctypes.byref(n)) == 1
    big = _shape(B=65536, T=65536, H=64, dk=128, dv=128)
    assert L.gdr_chunk_fwd_workspace(ctypes.byref(big), ctypes.byref(n)) == 2


FAKE = 0x10000  # a 64 KiB-aligned address that is never dereferenced


def _call_chunk(L, shape, **ptrs):
    p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, lam=None, b=None, w=None, h0=None,
             o=FAKE, hT=None, ws=None)
    p.update(ptrs)
    vp = ctypes.c_void_p
    sp = None if shape is None else ctypes.byref(shape)
    return L.gdr_chunk_fwd(sp, *(vp(p[n]) for n in
                                                 ("q", "k", "v", "g", "beta", "lam", "b", "w",
                                                  "h0", "o", "hT", "ws")),
                           ctypes.c_size_t(0), None)


def test_chunk_fwd_rejects_bad_arguments_synchronously(L):
    s = _shape()
    assert _call_chunk(L, s, q=None) == 1
    assert _call_chunk(L, s, o=None) == 1
    assert _call_chunk(L, s, g=None) == 1
    assert _call_chunk(L, s, beta=None) == 1                       # beta needed for GDN
    assert _call_chunk(L, _shape(flags=gdr.QMIX)) == 1              # lam missing
    assert _call_chunk(L, _shape(flags=gdr.ERASE_CHANNEL)) == 1     # b missing
    assert _call_chunk(L, _shape(flags=gdr.WRITE_CHANNEL)) == 1     # w missing
    assert _call_chunk(L, s, q=FAKE + 8) == 1                       # 16-byte alignment
    assert _call_chunk(L, s, h0=FAKE + 4) == 1
    assert _call_chunk(L, s, g=FAKE + 2) == 1
    assert _call_chunk(L, _shape(flags=gdr.DECAY_CHANNEL), g=FAKE + 4) == 1   # vector loads
    assert _call_chunk(L, _shape(dk=32)) == 2
    assert _call_chunk(L, _shape(dv=256)) == 2
    assert _call_chunk(L, _shape(H=0)) == 1
    assert _call_chunk(L, None) == 1


def test_recurrent_step_rejects_bad_arguments(L):
    vp = ctypes.c_void_p
    s = _shape(T=2)
    args = [vp(FAKE)] * 5 + [None, None, None, vp(FAKE), vp(FAKE), None]
    assert L.gdr_recurrent_step(ctypes.byref(s), *args) == 1        # T must be 1
    s = _shape(T=1)
    bad_state = [vp(FAKE)] * 5 + [None, None, None, None, vp(FAKE), None]
    assert L.gdr_recurrent_step(ctypes.byref(s), *bad_state) == 1
    s = _shape(T=1, dk=80)
    assert L.gdr_recurrent_step(ctypes.byref(s), *args) == 2


def test_workspace_rules(L):
    s = _shape()
    vp = ctypes.c_void_p
    # bf16 needs a workspace of at least 256 bytes, 16-byte aligned
    assert _call_chunk(L, s, ws=None) == 4
    p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, o=FAKE)
    args = [vp(p.get(n)) if p.get(n) else None for n in
            ("q", "k", "v", "g", "beta", "lam", "b", "w", "h0", "o", "hT")]
    assert L.gdr_chunk_fwd(ctypes.byref(s), *args, vp(FAKE), ctypes.c_size_t(128), None) == 4
    assert L.gdr_chunk_fwd(ctypes.byref(s), *args, vp(FAKE + 8), ctypes.c_size_t(256), None) == 4
    assert L.gdr_chunk_fwd_check(None, None, None) == 1


def test_gate_cumsum_rejects_bad_arguments(L):
    vp = ctypes.c_void_p
    assert L.gdr_gate_cumsum(1, 64, 4, 32, vp(FAKE), vp(FAKE), None) == 2   # chunk must be 64
    assert L.gdr_gate_cumsum(0, 64, 4, 64, vp(FAKE), vp(FAKE), None) == 1
    assert L.gdr_gate_cumsum(1, 64, 4, 64, None, vp(FAKE), None) == 1
    assert L.gdr_gate_cumsum(1, 64, 4, 64, vp(FAKE + 1), vp(FAKE), None) == 1


def test_binding_refuses_cpu_tensors(L):
    x = torch.zeros(1, 64, 1, 64)
    with pytest.raises(ValueError):
        gdr.chunk_fwd(x, x, x, torch.zeros(1, 64, 1), torch.zeros(1, 64, 1))


def test_product_code_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "gated_delta_rule_10_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\boracle\b\s*(import|\.)|from\s+oracle|import\s+oracle",
                                     text), f
                assert "gdr_oracle" not in text, f


def test_rmsnorm_gate_rejects_bad_arguments(L):
    vp, F = ctypes.c_void_p, ctypes.c_float

    def call(rows=4, dv=128, dtype=_binding.GDR_BF16, o=FAKE, z=FAKE + 0x4000, w=FAKE + 0x8000,
             eps=1e-6, y=FAKE + 0xC000):
        return L.gdr_rmsnorm_gate(rows, dv, dtype, vp(o) if o else None, vp(z) if z else None,
                                  vp(w) if w else None, F(eps), vp(y) if y else None, None)

    assert call(rows=0) == 0                       # nothing to do, nothing launched
    assert call(rows=0, o=None, z=None, w=None, y=None) == 0
    assert call(rows=-1) == 1
    assert call(dv=0) == 1
    assert call(dv=96) == 2
    assert call(dv=512) == 2
    assert call(dtype=5) == 1
    assert call(eps=-1e-6) == 1
    assert call(eps=float("inf")) == 1
    assert call(eps=float("nan")) == 1
    assert call(o=None) == 1
    assert call(w=None) == 1
    assert call(y=FAKE + 8) == 1                   # 16-byte alignment
    assert call(w=FAKE + 0x8004) == 1
    # 4 rows of 128 bf16 are 1 KiB: y overlapping o by part is refused
    assert call(y=FAKE + 0x200) == 1
    assert call(y=FAKE + 0x4000 - 0x200) == 1      # overlaps z
    assert call(rows=1 << 41) == 2


def test_value_beta_flag_rules(L):
    n = ctypes.c_size_t(7)
    BC = gdr.BETA_CHANNEL
    assert L.gdr_chunk_fwd_workspace(ctypes.byref(_shape(flags=BC)), ctypes.byref(n)) == 0
    # bf16: status words + one packet per chunk ([Q_gamma; K_gamma], K_tail, A_qk,
    # gamma_C, V, L fp32, beta bf16); fp32 needs none
    assert n.value == 256 + 3 * 64 * 64 * 2 + 8192 + 1024 + 2 * 64 * 64 * 2 + 64 * 64 * 4
    assert L.gdr_chunk_fwd_workspace(ctypes.byref(_shape(flags=BC, dtype=_binding.GDR_F32)),
                                     ctypes.byref(n)) == 0
    assert n.value == 0
    assert L.gdr_chunk_fwd_workspace_min(ctypes.byref(_shape(flags=BC)), ctypes.byref(n)) == 0
    assert n.value == 0
    for other in (gdr.DECAY_CHANNEL, gdr.ERASE_CHANNEL, gdr.WRITE_CHANNEL, gdr.QMIX):
        assert _call_chunk(L, _shape(flags=BC | other), b=FAKE, w=FAKE, lam=FAKE) == 2
    assert _call_chunk(L, _shape(flags=32)) == 1
    assert _call_chunk(L, _shape(flags=BC), beta=FAKE + 4) == 1     # 16-byte beta rows
    assert _call_chunk(L, _shape(flags=BC), beta=None) == 1
    big = _shape(B=1024, H=128, T=1, flags=BC)                       # grid y extent
    assert _call_chunk(L, big) == 2


def test_sequence_split_workspace_and_policy(L):
    n = ctypes.c_size_t(0)
    s = _shape(B=2, T=64 * 9 + 17, H=3, dk=128, dv=128)
    assert L.gdr_chunk_fwd_workspace_split(ctypes.byref(s), 1, ctypes.byref(n)) == 0
    two = 256 + 2 * 3 * 10 * 74752
    assert n.value == two
    assert L.gdr_chunk_fwd_workspace_split(ctypes.byref(s), 4, ctypes.byref(n)) == 0
    runs = 2 * 3 * 4
    al = lambda x: (x + 255) // 256 * 256
    assert n.value == al(two) + 2 * al(runs * 128 * 128 * 4) + al(runs * 128 * 128 * 4)
    assert L.gdr_chunk_fwd_workspace_split(ctypes.byref(s), 0, ctypes.byref(n)) == 1
    assert L.gdr_chunk_fwd_workspace_split(ctypes.byref(_shape(dtype=_binding.GDR_F32)), 2,
                                           ctypes.byref(n)) == 2
    assert L.gdr_chunk_fwd_workspace_split(ctypes.byref(_shape(flags=gdr.BETA_CHANNEL)), 2,
                                           ctypes.byref(n)) == 2
    # default policy: a long sequence with few heads is split, the benchmark shapes are not
    long_few = _shape(B=1, T=65536, H=4, dk=128, dv=128)
    assert L.gdr_chunk_fwd_workspace(ctypes.byref(long_few), ctypes.byref(n)) == 0
    plain = ctypes.c_size_t(0)
    L.gdr_chunk_fwd_workspace_split(ctypes.byref(long_few), 1, ctypes.byref(plain))
    assert n.value > plain.value
    L.gdr_chunk_fwd_workspace_split(ctypes.byref(long_few), 8, ctypes.byref(plain))
    assert n.value == plain.value                        # 8 x 4 x 4 = 128 CTAs, one wave
    for B, T, H in ((4, 4096, 16), (4, 8192, 16), (2, 16384, 32), (1, 65536, 32)):
        shp = _shape(B=B, T=T, H=H, dk=128, dv=128)
        L.gdr_chunk_fwd_workspace(ctypes.byref(shp), ctypes.byref(n))
        L.gdr_chunk_fwd_workspace_split(ctypes.byref(shp), 1, ctypes.byref(plain))
        assert n.value == plain.value
    # a forced split needs its workspace
    vp = ctypes.c_void_p
    assert L.gdr_chunk_fwd_split(ctypes.byref(s), 4, *(vp(FAKE),) * 5, None, None, None, None,
                                 vp(FAKE), None, vp(FAKE), ctypes.c_size_t(two), None) == 4
    assert L.gdr_chunk_fwd_split(ctypes.byref(s), 0, *(vp(FAKE),) * 5, None, None, None, None,
                                 vp(FAKE), None, vp(FAKE), ctypes.c_size_t(two), None) == 1
    # a forced split past the launch grid's extents is unsupported, not a failed launch:
    # B * segments (the split scan's grid z) and B * H (the run combination's grid y)
    for B, H, P in ((40000, 1, 2), (300, 300, 2)):
        big = _shape(B=B, T=64, H=H)
        assert L.gdr_chunk_fwd_split(ctypes.byref(big), P, *(vp(FAKE),) * 5, None, None, None,
                                     None, vp(FAKE), None, vp(FAKE), ctypes.c_size_t(1 << 40),
                                     None) == 2
    # one run stays the plain path at the same B * H
    big = _shape(B=300, T=64, H=300)
    n300 = ctypes.c_size_t(0)
    assert L.gdr_chunk_fwd_workspace_split(ctypes.byref(big), 1, ctypes.byref(n300)) == 0


def test_pipelined_forward_workspace_policy_and_argument_rules(L):
    n = ctypes.c_size_t(0)
    seg = ctypes.c_int(0)
    al = lambda x: (x + 255) // 256 * 256
    s = _shape(B=1, T=64 * 100 + 5, H=4, dk=128, dv=128)
    two = 256 + 4 * 101 * 74752
    assert L.gdr_chunk_fwd_workspace_pipelined(ctypes.byref(s), 4, ctypes.byref(n)) == 0
    assert n.value == al(two) + al(4 * 128 * 128 * 4) + al(4 * 4)
    assert L.gdr_chunk_fwd_workspace_pipelined(ctypes.byref(s), 0, ctypes.byref(n)) == 1
    assert L.gdr_chunk_fwd_workspace_pipelined(ctypes.byref(s), 65, ctypes.byref(n)) == 1
    assert L.gdr_chunk_fwd_workspace_pipelined(ctypes.byref(_shape(dtype=_binding.GDR_F32)), 2,
                                               ctypes.byref(n)) == 2
    assert L.gdr_chunk_fwd_workspace_pipelined(ctypes.byref(s), 2, None) == 1
    # policy: the Gated DeltaNet-2 prefill (B*H = 32, 1024 chunks) is pipelined in 8
    # segments, B*H = 64 (the transposed state pass takes 64 SMs) in up to 3 (one
    # per 32 chunks); workloads that the sequence split takes, that are short or
    # fp32 are not
    for (B, T, H, dt), want in (((1, 65536, 32, _binding.GDR_BF16), 8),
                                ((4, 4096, 16, _binding.GDR_BF16), 2),
                                ((4, 8192, 16, _binding.GDR_BF16), 3),
                                ((2, 16384, 32, _binding.GDR_BF16), 3),
                                ((8, 16384, 32, _binding.GDR_BF16), 1),
                                ((1, 65536, 4, _binding.GDR_BF16), 1),
                                ((1, 2048, 8, _binding.GDR_BF16), 1),
                                ((2, 8192, 16, _binding.GDR_BF16), 4),
                                ((1, 65536, 32, _binding.GDR_F32), 1)):
        shp = _shape(B=B, T=T, H=H, dk=128, dv=128, dtype=dt)
        assert L.gdr_chunk_fwd_pipeline_segments(ctypes.byref(shp), ctypes.byref(seg)) == 0
        assert seg.value == want, (B, T, H, dt)
    assert L.gdr_chunk_fwd_pipeline_segments(ctypes.byref(s), None) == 1
    assert L.gdr_chunk_fwd_pipeline_segments(ctypes.byref(_shape(dk=96)), ctypes.byref(seg)) == 2
    # argument errors return before anything is enqueued
    vp = ctypes.c_void_p

    def call(shape, segments, ws, ws_bytes, q=FAKE, hT=None):
        return L.gdr_chunk_fwd_pipelined(ctypes.byref(shape), segments, vp(q), *(vp(FAKE),) * 4,
                                         None, None, None, None, vp(FAKE),
                                         None if hT is None else vp(hT),
                                         None if ws is None else vp(ws), ctypes.c_size_t(ws_bytes),
                                         None, None)
    L.gdr_chunk_fwd_workspace_pipelined(ctypes.byref(s), 4, ctypes.byref(n))
    full = n.value
    assert call(s, 4, FAKE, full - 1) == 4
    assert call(s, 4, None, full) == 4
    assert call(s, 4, FAKE + 8, full) == 4
    assert call(s, 0, FAKE, full) == 1
    assert call(s, 4, FAKE, full, q=None) == 1
    assert call(s, 4, FAKE, full, hT=FAKE + 4) == 1
    assert call(_shape(dtype=_binding.GDR_F32), 2, FAKE, full) == 2


def _bwd_ws(fn, **kw):
    n = ctypes.c_size_t(0)
    st = fn(ctypes.byref(_shape(**kw)), ctypes.byref(n))
    return st, n.value


@pytest.mark.parametrize("name", ["gdr_chunk_bwd_workspace", "gdr_token_bwd_workspace"])
def test_backward_workspace_queries(L, name):
    """The backwards' workspace sizes: a fixed head (status words), then a share
    per 64-token chunk of every (batch, head) sequence (the token-order one also
    holds one chunk of token states per sequence), so they grow by equal steps
    in B and H, a ragged tail costs a whole chunk, and invalid shapes are
    refused like the forward's."""
    fn = getattr(L, name)
    st, one = _bwd_ws(fn, dk=128, dv=128)
    assert st == 0 and one > 0
    sizes = [_bwd_ws(fn, B=b, dk=128, dv=128)[1] for b in (1, 2, 3)]
    assert sizes[1] - sizes[0] == sizes[2] - sizes[1] > 0
    assert _bwd_ws(fn, H=3, dk=128, dv=128)[1] == sizes[2]
    assert _bwd_ws(fn, T=65, dk=128, dv=128)[1] == _bwd_ws(fn, T=128, dk=128, dv=128)[1]
    step_t = _bwd_ws(fn, T=128, dk=128, dv=128)[1] - one   # one more chunk
    if name == "gdr_chunk_bwd_workspace":
        assert step_t == sizes[1] - sizes[0]                 # everything is per chunk
    else:
        assert 0 < step_t < sizes[1] - sizes[0]              # a checkpoint, not a sequence
    # wider states take more per chunk
    assert _bwd_ws(fn, dk=64, dv=64)[1] < one
    # refusals: no output pointer, no shape, unsupported width, empty sequence
    n = ctypes.c_size_t(0)
    assert fn(ctypes.byref(_shape()), None) == 1
    assert fn(None, ctypes.byref(n)) == 1
    assert _bwd_ws(fn, dk=96)[0] == 2
    assert _bwd_ws(fn, T=0)[0] == 1


def test_chunk_backward_workspace_per_chunk(L):
    """gdr.h states about 0.79 MB of chunk-backward workspace per chunk at
    d_k = d_v = 128 (records, scratch, the states and their gradients)."""
    _, a = _bwd_ws(L.gdr_chunk_bwd_workspace, B=1, T=64 * 64, dk=128, dv=128)
    _, b = _bwd_ws(L.gdr_chunk_bwd_workspace, B=2, T=64 * 64, dk=128, dv=128)
    per_chunk = (b - a) / 64
    assert 0.75e6 < per_chunk < 0.83e6


def test_value_beta_backward_workspace_is_the_token_order_one(L):
    """The per-value-channel write strength has no chunk backward of its own:
    both queries give the token-order backward's workspace for it."""
    bc = gdr.BETA_CHANNEL
    for dk, dv in ((64, 64), (128, 128), (64, 128)):
        st1, a = _bwd_ws(L.gdr_chunk_bwd_workspace, T=1000, dk=dk, dv=dv, flags=bc)
        st2, b = _bwd_ws(L.gdr_token_bwd_workspace, T=1000, dk=dk, dv=dv, flags=bc)
        assert st1 == st2 == 0 and a == b > 0
