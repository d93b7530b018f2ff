"""The C ABI without a GPU: the library loads, exports what include/kda.h declares,
the header compiles as C, and argument validation / the alias guard reject bad calls
before anything is enqueued (no CUDA call is made on these paths)."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def native():
    from kimi_delta_attention_09_gb300 import build
    build.build()
    from kimi_delta_attention_09_gb300 import _native
    return _native


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    assert "kda_chunk_prefill" in syms and "kda_recurrent_decode" in syms
    assert len(syms) >= 5


def test_library_exports_every_declared_symbol(native):
    out = subprocess.run(["nm", "-D", "--defined-only", native.LIB_PATH], check=True,
                         capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(kda_\w+)", out))
    for s in declared_symbols():
        assert s in exported, s
        assert hasattr(native.lib, s)
    assert set(native.EXPORTED) == set(declared_symbols())


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "kda.h"\nint main(void) { return kda_abi_version() == '
                   'KDA_ABI_VERSION ? KDA_OK : KDA_ERR_CUDA; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I" + os.path.dirname(HEADER), "-c", str(src), "-o",
                    str(tmp_path / "use.o")], check=True)


def test_status_strings(native):
    assert native.lib.kda_abi_version() == 5
    for code, name in [(0, "KDA_OK"), (-1, "KDA_ERR_INVALID_ARG"), (-2, "KDA_ERR_UNSUPPORTED"),
                       (-3, "KDA_ERR_ALIAS"), (-4, "KDA_ERR_CUDA"), (-5, "KDA_ERR_TIMEOUT")]:
        assert native.status_string(code) == name
    assert native.status_string(7) == "KDA_ERR_UNKNOWN"


# Fake, never-dereferenced device addresses: validation must decide from the
# addresses and sizes alone.  Every call below is built to FAIL validation (or to
# have nothing to do), so no kernel is ever launched on these addresses.
BASE = 1 << 40


def _prefill(native, **kw):
    T, N, H, K, V, es = kw.get("T", 100), kw.get("N", 2), 2, 64, 64, 2
    a = dict(q=BASE, k=BASE + (1 << 24), v=BASE + (2 << 24), g=BASE + (3 << 24),
             beta=BASE + (4 << 24), scale=0.125, init=BASE + (5 << 24), cu=BASE + (6 << 24),
             out=BASE + (7 << 24), final=BASE + (8 << 24), T=T, N=N, H=H, K=K, V=V, dtype=1,
             out_dtype=1)
    a.update(kw)
    vp = ctypes.c_void_p
    return native.lib.kda_chunk_prefill(
        vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["g"]), vp(a["beta"]), a["scale"],
        vp(a["init"]), vp(a["cu"]), vp(a["out"]), vp(a["final"]), a["T"], a["N"], a["H"],
        a["K"], a["V"], a["dtype"], a["out_dtype"], a.get("flags", 0), None)


def _decode(native, **kw):
    a = dict(q=BASE, k=BASE + (1 << 24), v=BASE + (2 << 24), g=BASE + (3 << 24),
             beta=BASE + (4 << 24), scale=0.125, pool=BASE + (1 << 32), idx=BASE + (6 << 24),
             out=BASE + (7 << 24), N=4, S=8, H=2, K=128, V=128, dtype=1, out_dtype=1)
    a.update(kw)
    vp = ctypes.c_void_p
    return native.lib.kda_recurrent_decode(
        vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["g"]), vp(a["beta"]), a["scale"],
        vp(a["pool"]), vp(a["idx"]), vp(a["out"]), a["N"], a["S"], a["H"], a["K"], a["V"],
        a["dtype"], a["out_dtype"], a.get("flags", 0), None)


def test_unknown_option_bits_are_rejected(native):
    # every call is built to fail on its flags alone (sizes and addresses are valid)
    assert _prefill(native, flags=2) == native.KDA_ERR_INVALID_ARG
    assert _prefill(native, flags=native.KDA_FLAG_QK_L2NORM | 8) == native.KDA_ERR_INVALID_ARG
    assert _decode(native, flags=4) == native.KDA_ERR_INVALID_ARG
    assert _decode_bf16_state(native, flags=-1) == native.KDA_ERR_INVALID_ARG
    assert _prefill_paged(native, flags=16) == native.KDA_ERR_INVALID_ARG


def test_prefill_argument_validation(native):
    assert _prefill(native, q=None) == native.KDA_ERR_INVALID_ARG
    assert _prefill(native, cu=None) == native.KDA_ERR_INVALID_ARG
    assert _prefill(native, out=BASE + (7 << 24) + 8) == native.KDA_ERR_INVALID_ARG  # misaligned
    assert _prefill(native, T=-1) == native.KDA_ERR_INVALID_ARG
    assert _prefill(native, H=0) == native.KDA_ERR_INVALID_ARG
    assert _prefill(native, scale=float("nan")) == native.KDA_ERR_INVALID_ARG
    assert _prefill(native, K=96) == native.KDA_ERR_UNSUPPORTED
    assert _prefill(native, V=256) == native.KDA_ERR_UNSUPPORTED
    assert _prefill(native, dtype=5) == native.KDA_ERR_UNSUPPORTED
    assert _prefill(native, out_dtype=2) == native.KDA_ERR_UNSUPPORTED
    assert _prefill(native, N=0) == native.KDA_OK            # nothing to do, nothing enqueued


def test_prefill_alias_guard(native):
    # out overlapping q, v, g, beta or cu_seqlens
    for key in ("q", "v", "g", "beta", "cu"):
        base = {"q": BASE, "v": BASE + (2 << 24), "g": BASE + (3 << 24),
                "beta": BASE + (4 << 24), "cu": BASE + (6 << 24)}[key]
        assert _prefill(native, out=base) == native.KDA_ERR_ALIAS, key
    # an fp32 out is twice as long as a bf16 one: 2 bytes past the bf16 end of out
    # would be free for bf16 but overlaps for fp32 (out is [100, 2, 64])
    bf16_end = BASE + (9 << 24)
    assert _prefill(native, out=bf16_end - 100 * 2 * 64 * 4 + 16, final=bf16_end,
                    out_dtype=0) == native.KDA_ERR_ALIAS
    # final_state overlapping k (partial overlap, not just equal start)
    assert _prefill(native, final=BASE + (1 << 24) + 4096) == native.KDA_ERR_ALIAS
    # final_state partially overlapping init_state is rejected ...
    assert _prefill(native, final=BASE + (5 << 24) + 16) == native.KDA_ERR_ALIAS
    # ... out overlapping final_state is rejected ...
    assert _prefill(native, out=BASE + (8 << 24) + 64) == native.KDA_ERR_ALIAS


def _prefill_paged(native, **kw):
    a = dict(q=BASE, k=BASE + (1 << 24), v=BASE + (2 << 24), g=BASE + (3 << 24),
             beta=BASE + (4 << 24), scale=0.125, pool=BASE + (1 << 32), idx=BASE + (5 << 24),
             cu=BASE + (6 << 24), out=BASE + (7 << 24), T=100, N=2, S=8, H=2, K=128, V=128,
             dtype=1, out_dtype=0)
    a.update(kw)
    vp = ctypes.c_void_p
    return native.lib.kda_chunk_prefill_paged(
        vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["g"]), vp(a["beta"]), a["scale"],
        vp(a["pool"]), vp(a["idx"]), vp(a["cu"]), vp(a["out"]), a["T"], a["N"], a["S"], a["H"],
        a["K"], a["V"], a["dtype"], a["out_dtype"], a.get("flags", 0), None)


def test_paged_prefill_validation_and_alias(native):
    assert _prefill_paged(native, idx=None) == native.KDA_ERR_INVALID_ARG
    assert _prefill_paged(native, pool=None) == native.KDA_ERR_INVALID_ARG
    assert _prefill_paged(native, S=-1) == native.KDA_ERR_INVALID_ARG
    assert _prefill_paged(native, K=96) == native.KDA_ERR_UNSUPPORTED
    assert _prefill_paged(native, N=0) == native.KDA_OK
    assert _prefill_paged(native, out=BASE + (1 << 32) + 512) == native.KDA_ERR_ALIAS
    assert _prefill_paged(native, pool=BASE + (2 << 24)) == native.KDA_ERR_ALIAS
    assert _prefill_paged(native, idx=BASE + (1 << 32) + 64) == native.KDA_ERR_ALIAS


def test_decode_argument_validation_and_alias(native):
    assert _decode(native, idx=None) == native.KDA_ERR_INVALID_ARG
    assert _decode(native, pool=None) == native.KDA_ERR_INVALID_ARG
    assert _decode(native, K=32) == native.KDA_ERR_UNSUPPORTED
    assert _decode(native, N=-1) == native.KDA_ERR_INVALID_ARG
    assert _decode(native, N=0) == native.KDA_OK
    # out inside the pool, pool overlapping an input
    assert _decode(native, out=BASE + (1 << 32) + 4096) == native.KDA_ERR_ALIAS
    assert _decode(native, pool=BASE + (3 << 24)) == native.KDA_ERR_ALIAS
    assert _decode(native, idx=BASE + (1 << 32) + 64) == native.KDA_ERR_ALIAS


def _decode_bf16_state(native, **kw):
    a = dict(q=BASE, k=BASE + (1 << 24), v=BASE + (2 << 24), g=BASE + (3 << 24),
             beta=BASE + (4 << 24), scale=0.125, pool=BASE + (1 << 32), idx=BASE + (6 << 24),
             out=BASE + (7 << 24), N=4, S=8, H=2, K=128, V=128, dtype=1, out_dtype=1)
    a.update(kw)
    vp = ctypes.c_void_p
    return native.lib.kda_recurrent_decode_bf16_state(
        vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["g"]), vp(a["beta"]), a["scale"],
        vp(a["pool"]), vp(a["idx"]), vp(a["out"]), a["N"], a["S"], a["H"], a["K"], a["V"],
        a["dtype"], a["out_dtype"], a.get("flags", 0), None)


def test_decode_bf16_state_argument_validation_and_alias(native):
    assert _decode_bf16_state(native, idx=None) == native.KDA_ERR_INVALID_ARG
    assert _decode_bf16_state(native, pool=None) == native.KDA_ERR_INVALID_ARG
    assert _decode_bf16_state(native, pool=BASE + (1 << 32) + 8) == native.KDA_ERR_INVALID_ARG
    assert _decode_bf16_state(native, V=96) == native.KDA_ERR_UNSUPPORTED
    assert _decode_bf16_state(native, dtype=7) == native.KDA_ERR_UNSUPPORTED
    assert _decode_bf16_state(native, N=0) == native.KDA_OK
    # the bf16 pool spans S H K V * 2 bytes: its last 16 bytes still alias the output
    pool_bytes = 8 * 2 * 128 * 128 * 2
    assert _decode_bf16_state(native, out=BASE + (1 << 32) + pool_bytes - 16) == native.KDA_ERR_ALIAS
    assert _decode_bf16_state(native, pool=BASE + (3 << 24)) == native.KDA_ERR_ALIAS
    assert _decode_bf16_state(native, idx=BASE + (1 << 32) + 64) == native.KDA_ERR_ALIAS


def test_binding_refuses_missing_library(tmp_path, monkeypatch):
    """No fallback: the binding raises when libkda.so is absent."""
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "kda_native_copy", os.path.join(ROOT, "kimi_delta_attention_09_gb300", "_native.py"))
    mod = importlib.util.module_from_spec(spec)
    monkeypatch.setattr(os.path, "exists",
                        lambda p, _e=os.path.exists: False if p.endswith("libkda.so") else _e(p))
    with pytest.raises(RuntimeError, match="not built"):
        spec.loader.exec_module(mod)


def _prefill_ws(native, ws, ws_bytes, **kw):
    """kda_chunk_prefill_ws with the argument set of _prefill (K = V = 128, bf16 by
    default: the shapes that need a workspace)."""
    a = dict(q=BASE, k=BASE + (1 << 24), v=BASE + (2 << 24), g=BASE + (3 << 24),
             beta=BASE + (4 << 24), scale=0.125, init=BASE + (5 << 24), cu=BASE + (6 << 24),
             out=BASE + (7 << 24), final=BASE + (8 << 24), T=100, N=2, H=2, K=128, V=128,
             dtype=1, out_dtype=1)
    a.update(kw)
    vp = ctypes.c_void_p
    return native.lib.kda_chunk_prefill_ws(
        vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["g"]), vp(a["beta"]), a["scale"],
        vp(a["init"]), vp(a["cu"]), vp(a["out"]), vp(a["final"]), a["T"], a["N"], a["H"],
        a["K"], a["V"], a["dtype"], a["out_dtype"], vp(ws), ws_bytes, a.get("flags", 0), None)


def test_workspace_query_is_zero_without_the_tensor_core_kernel(native):
    q = native.lib.kda_chunk_prefill_workspace_bytes
    assert q(2, 2, 128, 128, 0) == 0      # fp32 inputs
    assert q(2, 2, 64, 128, 1) == 0       # K = 64
    assert q(2, 2, 128, 64, 1) == 0       # V = 64
    assert q(0, 2, 128, 128, 1) == 0      # no sequences
    # a 256-byte status header, then whole rings of 8 records of 66,816 B (one per cluster)
    n = q(2, 2, 128, 128, 1)
    assert n > 256 and (n - 256) % (8 * 66816) == 0


def test_prefill_ws_validation_and_alias(native):
    need = native.lib.kda_chunk_prefill_workspace_bytes(2, 2, 128, 128, 1)
    ws = BASE + (1 << 36)
    # the shared argument checks come first
    assert _prefill_ws(native, ws, need, q=None) == native.KDA_ERR_INVALID_ARG
    assert _prefill_ws(native, ws, need, K=96) == native.KDA_ERR_UNSUPPORTED
    assert _prefill_ws(native, ws, need, out=BASE) == native.KDA_ERR_ALIAS
    assert _prefill_ws(native, None, 0, N=0) == native.KDA_OK
    # the workspace itself: missing, too small, misaligned
    assert _prefill_ws(native, None, 0) == native.KDA_ERR_INVALID_ARG
    assert _prefill_ws(native, ws, need - 16) == native.KDA_ERR_INVALID_ARG
    assert _prefill_ws(native, ws + 8, need) == native.KDA_ERR_INVALID_ARG
    # ... and overlapping any input or output (partially, at either end)
    assert _prefill_ws(native, BASE + (1 << 24) - need + 16, need) == native.KDA_ERR_ALIAS   # k
    assert _prefill_ws(native, BASE + (7 << 24) + 4096, need) == native.KDA_ERR_ALIAS       # out
    assert _prefill_ws(native, BASE + (8 << 24) - 16, need) == native.KDA_ERR_ALIAS         # final
    assert _prefill_ws(native, BASE + (6 << 24), need) == native.KDA_ERR_ALIAS              # cu_seqlens


def test_prefill_noalloc_validation(native):
    vp = ctypes.c_void_p

    def call(**kw):
        a = dict(q=BASE, k=BASE + (1 << 24), v=BASE + (2 << 24), g=BASE + (3 << 24),
                 beta=BASE + (4 << 24), scale=0.125, init=BASE + (5 << 24), cu=BASE + (6 << 24),
                 out=BASE + (7 << 24), final=BASE + (8 << 24), T=100, N=2, H=2, K=128, V=128,
                 dtype=1, out_dtype=1)
        a.update(kw)
        return native.lib.kda_chunk_prefill_noalloc(
            vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["g"]), vp(a["beta"]), a["scale"],
            vp(a["init"]), vp(a["cu"]), vp(a["out"]), vp(a["final"]), a["T"], a["N"], a["H"],
            a["K"], a["V"], a["dtype"], a["out_dtype"], None)

    assert call(q=None) == native.KDA_ERR_INVALID_ARG
    assert call(scale=float("inf")) == native.KDA_ERR_INVALID_ARG
    assert call(V=96) == native.KDA_ERR_UNSUPPORTED
    assert call(final=BASE + (1 << 24)) == native.KDA_ERR_ALIAS
    assert call(N=0) == native.KDA_OK


def test_paged_prefill_ws_validation_and_alias(native):
    vp = ctypes.c_void_p
    need = native.lib.kda_chunk_prefill_workspace_bytes(2, 2, 128, 128, 1)

    def call(ws, ws_bytes, **kw):
        a = dict(q=BASE, k=BASE + (1 << 24), v=BASE + (2 << 24), g=BASE + (3 << 24),
                 beta=BASE + (4 << 24), scale=0.125, pool=BASE + (1 << 32), idx=BASE + (5 << 24),
                 cu=BASE + (6 << 24), out=BASE + (7 << 24), T=100, N=2, S=8, H=2, K=128, V=128,
                 dtype=1, out_dtype=0)
        a.update(kw)
        return native.lib.kda_chunk_prefill_paged_ws(
            vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["g"]), vp(a["beta"]), a["scale"],
            vp(a["pool"]), vp(a["idx"]), vp(a["cu"]), vp(a["out"]), a["T"], a["N"], a["S"],
            a["H"], a["K"], a["V"], a["dtype"], a["out_dtype"], vp(ws), ws_bytes, a.get("flags", 0), None)

    ws = BASE + (1 << 36)
    assert call(ws, need, idx=None) == native.KDA_ERR_INVALID_ARG
    assert call(ws, need, out=BASE + (1 << 32)) == native.KDA_ERR_ALIAS      # out over the pool
    assert call(None, 0) == native.KDA_ERR_INVALID_ARG                       # workspace needed
    assert call(ws, need - 16) == native.KDA_ERR_INVALID_ARG
    assert call(BASE + (1 << 32) + 64, need) == native.KDA_ERR_ALIAS         # workspace over the pool
    assert call(BASE + (5 << 24), need) == native.KDA_ERR_ALIAS              # ... over state_idx
    assert call(None, 0, N=0) == native.KDA_OK


def _conv(native, prompt=True, **kw):
    vp = ctypes.c_void_p
    a = dict(x=BASE, w=BASE + (1 << 24), b=BASE + (2 << 24), st=BASE + (3 << 24), idx=BASE + (4 << 24),
             cu=BASE + (5 << 24), out=BASE + (6 << 24), T=100, N=2, S=4, D=64, W=4, dtype=1,
             out_dtype=0, act=1)
    a.update(kw)
    if prompt:
        return native.lib.kda_causal_conv1d_fwd(
            vp(a["x"]), vp(a["w"]), vp(a["b"]), vp(a["st"]), vp(a["idx"]), vp(a["cu"]), vp(a["out"]),
            a["T"], a["N"], a["S"], a["D"], a["W"], a["dtype"], a["out_dtype"], a["act"], None)
    return native.lib.kda_causal_conv1d_update(
        vp(a["x"]), vp(a["w"]), vp(a["b"]), vp(a["st"]), vp(a["idx"]), vp(a["out"]),
        a["N"], a["S"], a["D"], a["W"], a["dtype"], a["out_dtype"], a["act"], None)


def test_conv_validation_and_alias(native):
    for prompt in (True, False):
        assert _conv(native, prompt, W=0) == native.KDA_ERR_INVALID_ARG
        assert _conv(native, prompt, W=5) == native.KDA_ERR_INVALID_ARG
        assert _conv(native, prompt, D=66) == native.KDA_ERR_INVALID_ARG      # not a multiple of 4
        assert _conv(native, prompt, act=2) == native.KDA_ERR_INVALID_ARG
        assert _conv(native, prompt, dtype=7) == native.KDA_ERR_UNSUPPORTED
        assert _conv(native, prompt, x=None) == native.KDA_ERR_INVALID_ARG
        assert _conv(native, prompt, w=None) == native.KDA_ERR_INVALID_ARG
        assert _conv(native, prompt, idx=None) == native.KDA_ERR_INVALID_ARG  # taps need slots
        assert _conv(native, prompt, out=BASE + 8) == native.KDA_ERR_INVALID_ARG   # misaligned
        assert _conv(native, prompt, N=0) == native.KDA_OK
        assert _conv(native, prompt, out=BASE + 64) == native.KDA_ERR_ALIAS    # out over x
        assert _conv(native, prompt, st=BASE + (6 << 24) + 16) == native.KDA_ERR_ALIAS   # taps over out
        assert _conv(native, prompt, st=BASE + (1 << 24) - 64) == native.KDA_ERR_ALIAS   # taps over weight
    assert _conv(native, True, cu=None) == native.KDA_ERR_INVALID_ARG
