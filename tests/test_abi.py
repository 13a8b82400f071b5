"""CPU checks of the C ABI: libkda builds, loads without a GPU, exports every
symbol include/kda.h declares, and rejects bad arguments on the host before
anything is launched (no CUDA call is reached by these cases)."""
import ctypes
import os
import re

import numpy as np
import pytest

from kda_linear_attention_bounded_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    path = kbuild.build()
    from kda_linear_attention_bounded_gb300 import _binding
    return _binding.load()


def declared_symbols():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"KDA_API\s+[\w\s\*]*?\b(kda_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    syms = declared_symbols()
    for name in ("kda_chunk_prefill", "kda_recurrent_verify", "kda_workspace_size", "kda_status_string"):
        assert name in syms


def test_binding_constants_match_the_header():
    from kda_linear_attention_bounded_gb300 import _binding as b
    defines = re.findall(r"#define\s+(KDA_[A-Z_0-9]+)\s+\(?(-?\d+)u?\)?", open(HEADER).read())
    assert len(defines) >= 11
    for name, value in defines:
        assert getattr(b, name) == int(value), name


def test_every_declared_symbol_is_exported(lib):
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, f"not exported: {missing}"


def test_status_strings(lib):
    from kda_linear_attention_bounded_gb300 import _binding as b
    for code in range(0, 5):
        assert b.status_string(code).startswith("KDA_")
    assert "unknown" in b.status_string(99)


def test_workspace_size(lib):
    n = lib.kda_workspace_size()
    assert n > 0 and n % 256 == 0


# ---- host-side validation (fake, aligned device addresses; never dereferenced) ----
FAKE = 0x10000000
P = ctypes.c_void_p


def _prefill(lib, *, cu=(0, 4), H=2, lb=-5.0, scale=0.1, ws=FAKE, ws_bytes=1024, stride=256, flags=0,
             q=FAKE, final=FAKE, pool=None, slots=None, nslots=0, norm=None, conv=None):
    cu_host = np.array(cu, np.int32)
    return lib.kda_chunk_prefill(P(q), P(FAKE), P(FAKE), stride, P(FAKE), stride, P(FAKE), H, P(FAKE), P(FAKE),
                                 lb, scale, P(FAKE), cu_host.ctypes.data_as(P), len(cu) - 1, H, P(pool), nslots,
                                 P(slots), flags, P(FAKE), stride, norm, conv, P(final), P(ws), ws_bytes, None)


def _verify(lib, *, B=2, T=8, H=2, lb=-5.0, ws=FAKE, pool=FAKE, inter=FAKE, norm=None, conv=None):
    return lib.kda_recurrent_verify(P(FAKE), P(FAKE), P(FAKE), H * 128, P(FAKE), H * 128, P(FAKE), H, P(FAKE),
                                    P(FAKE), lb, 0.1, B, T, H, P(pool), 4, P(FAKE), P(FAKE), H * 128, norm, conv,
                                    P(inter), P(ws), 1024, None)


def _conv(weight=FAKE, act=1, pool=FAKE, dense=None, steps=FAKE):
    from kda_linear_attention_bounded_gb300._binding import _ShortConvC
    return ctypes.byref(_ShortConvC(weight, act, pool, dense, steps))


def _norm(gate=FAKE, stride=256, weight=FAKE, eps=1e-6, rstd=None):
    from kda_linear_attention_bounded_gb300._binding import _OutputNormC
    return ctypes.byref(_OutputNormC(gate, stride, weight, eps, rstd))


def test_prefill_rejects_bad_arguments(lib):
    assert _prefill(lib, ws=None) == 3
    assert _prefill(lib, ws=FAKE + 16) == 3           # misaligned workspace
    assert _prefill(lib, ws_bytes=16) == 3
    assert _prefill(lib, cu=(0, 5, 3)) == 1            # decreasing cu_seqlens
    assert _prefill(lib, cu=(1, 5)) == 1               # not starting at 0
    assert _prefill(lib, lb=-20.0) == 2                # outside the supported bound
    assert _prefill(lib, lb=0.5) == 2
    assert _prefill(lib, lb=float("nan")) == 2
    assert _prefill(lib, scale=float("inf")) == 2
    assert _prefill(lib, stride=100) == 1              # stride below H*128
    assert _prefill(lib, stride=260) == 1              # stride not a multiple of 8
    assert _prefill(lib, q=FAKE + 2) == 1              # misaligned pointer
    assert _prefill(lib, q=None) == 1
    assert _prefill(lib, final=None) == 1              # dense final state required
    assert _prefill(lib, flags=1) == 1                 # pool + slot ids required
    assert _prefill(lib, flags=32) == 1                # unknown flag
    assert _prefill(lib, flags=4 | 8) == 1             # two execution paths forced
    assert _prefill(lib, flags=4 | 16) == 1
    assert _prefill(lib, flags=8 | 16) == 1
    assert _prefill(lib, flags=8, lb=-6.0, ws_bytes=1 << 30) == 2   # the fused path takes lower_bound >= -5 only
    assert _prefill(lib, H=0) == 1
    assert _prefill(lib, cu=(0,)) == 0                 # no sequences: nothing to do
    # valid arguments but a workspace without room for the chunk blocks
    need = lib.kda_prefill_workspace_size(4, 1, 2)
    scratch = 2 * 128 * 128 * 4                        # one sequence x two heads of fp32 state
    assert _prefill(lib, ws_bytes=need - scratch - 256) == 3
    # forced split state passes with the blocks but without the scratch states
    assert _prefill(lib, flags=16, ws_bytes=need - scratch) == 3


def test_prefill_workspace_size(lib):
    lib.kda_prefill_workspace_size.restype = ctypes.c_size_t
    lib.kda_prefill_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int]
    block, state = 74240, 128 * 128 * 4
    # header + (floor(T / 64) + num_seqs) chunks x H blocks (an upper bound of sum ceil(len / 64)) + the fp32
    # states of min(num_seqs x H, 96) (sequence, head) pairs handed between segments of split state passes
    assert lib.kda_prefill_workspace_size(2048 * 8, 8, 16) == 1024 + (256 + 8) * 16 * block + 96 * state
    assert lib.kda_prefill_workspace_size(0, 3, 2) == 1024 + 3 * 2 * block + 6 * state
    assert lib.kda_prefill_workspace_size(130, 1, 1) == 1024 + 3 * block + state
    assert lib.kda_prefill_workspace_size(-1, 1, 1) == 0
    assert lib.kda_prefill_workspace_size(10, 1, 0) == 0


def test_verify_rejects_bad_arguments(lib):
    assert _verify(lib, ws=None) == 3
    assert _verify(lib, T=0) == 1
    assert _verify(lib, T=65) == 1
    assert _verify(lib, B=-1) == 1
    assert _verify(lib, lb=-11.0) == 2
    assert _verify(lib, pool=None) == 1
    assert _verify(lib, inter=None) == 1
    assert _verify(lib, B=0) == 0                      # no requests: nothing to do


def _spec_step(lib, *, cu=(0, 4), B=2, T=8, H=2, pre=True, spec=True, pre_stride=256, spec_stride=256,
               ns_idx=FAKE, s_idx=FAKE, n_out=100, ws_bytes=None, lb=-5.0, norm=None, conv=None, flags=0):
    from kda_linear_attention_bounded_gb300._binding import TokenTensors
    cu_host = np.array(cu, np.int32)
    ws_bytes = lib.kda_prefill_workspace_size(int(cu[-1]), len(cu) - 1, H) if ws_bytes is None else ws_bytes
    tp = TokenTensors(FAKE, FAKE, FAKE, pre_stride, FAKE, pre_stride, FAKE, H)
    ts = TokenTensors(FAKE, FAKE, FAKE, spec_stride, FAKE, spec_stride, FAKE, H)
    return lib.kda_spec_step(ctypes.byref(tp) if pre else None, P(FAKE), cu_host.ctypes.data_as(P), len(cu) - 1,
                             None, flags, P(FAKE), ctypes.byref(ts) if spec else None, B, T, P(FAKE), P(FAKE), P(FAKE),
                             P(FAKE), lb, 0.1, H, P(FAKE), 4, P(FAKE), H * 128, n_out, norm, conv, P(ns_idx),
                             P(s_idx), P(FAKE), ws_bytes, None)


def test_spec_step_rejects_bad_arguments(lib):
    # every check of both segments runs before anything is launched
    assert _spec_step(lib, pre=False) == 1            # a prefill segment without its tensors
    assert _spec_step(lib, spec=False) == 1           # a verify segment without its tensors
    assert _spec_step(lib, pre_stride=100) == 1
    assert _spec_step(lib, spec_stride=260) == 1
    assert _spec_step(lib, T=0) == 1
    assert _spec_step(lib, cu=(0, 5, 3)) == 1
    assert _spec_step(lib, ns_idx=None) == 1          # prefill tokens need their output rows
    assert _spec_step(lib, s_idx=None) == 1           # and so do the verify tokens
    assert _spec_step(lib, n_out=-1) == 1
    assert _spec_step(lib, lb=-11.0) == 2
    assert _spec_step(lib, ws_bytes=256) == 3         # no room for the prefill's chunk blocks
    assert _spec_step(lib, cu=(0,), B=0, pre=False, spec=False, ns_idx=None, s_idx=None) == 0   # empty step


def test_output_norm_is_checked_on_the_host(lib):
    # every call rejects a bad norm descriptor before launching anything
    for bad in (_norm(gate=None), _norm(gate=FAKE + 2), _norm(stride=100), _norm(stride=260), _norm(weight=None),
                _norm(weight=FAKE + 4), _norm(eps=-1.0), _norm(eps=float("nan")), _norm(rstd=FAKE + 2)):
        assert _prefill(lib, norm=bad, ws_bytes=lib.kda_prefill_workspace_size(4, 1, 2)) == 1
        assert _verify(lib, norm=bad) == 1
        assert _spec_step(lib, norm=bad) == 1
    assert _prefill(lib, cu=(0,), norm=_norm(gate=None)) == 0    # nothing to do: the norm is not looked at


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from kda_linear_attention_bounded_gb300 import _binding as b
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        b.load()


def test_commit_rejects_bad_arguments(lib):
    c = lambda **kw: lib.kda_commit_accepted(P(kw.get("pool", FAKE)), 4, P(FAKE), P(FAKE), P(kw.get("inter", FAKE)),
                                             kw.get("conv"), kw.get("B", 2), kw.get("T", 8), 2, P(kw.get("ws", FAKE)),
                                             1024, None)
    assert c(ws=None) == 3
    assert c(pool=None) == 1
    assert c(pool=FAKE + 4) == 1
    assert c(inter=None) == 1
    assert c(T=0) == 1
    assert c(T=65) == 1
    assert c(B=0) == 0
    assert c(conv=_conv(pool=None)) == 1
    assert c(conv=_conv(steps=FAKE + 8)) == 1


def test_short_conv_is_checked_on_the_host(lib):
    for bad in (_conv(weight=None), _conv(weight=FAKE + 4), _conv(act=2), _conv(pool=None), _conv(steps=None),
                _conv(pool=FAKE + 2)):
        assert _verify(lib, conv=bad) == 1
        assert _spec_step(lib, conv=bad, cu=(0,), pre=False) == 1
