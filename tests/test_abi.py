"""The C ABI without a GPU: the library builds, loads, exports every symbol that
include/rlk.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rlk.h")

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3
FAKE = ctypes.c_void_p(0x100000)      # 16- and 256-byte aligned, never dereferenced
MISALIGNED = ctypes.c_void_p(0x100002)


@pytest.fixture(scope="module")
def lib():
    from deterministic_token_logprob_gb300 import build
    build.build()
    import deterministic_token_logprob_gb300 as rlk
    return rlk.lib()   # the binding declares argtypes / restype of every entry point


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rlk_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("rlk_linear_logp_fwd", "rlk_linear_logp_bwd", "rlk_lse_merge",
              "rlk_linear_logp_fwd_workspace", "rlk_linear_logp_bwd_workspace"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_only_declared_symbols_are_exported(lib):
    import subprocess
    from deterministic_token_logprob_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    rlk_syms = {s for s in exported if s.startswith("rlk_")}
    assert rlk_syms == set(declared_functions())


def test_version_and_status_strings(lib):
    assert lib.rlk_version().decode().startswith("rlk ")
    assert lib.rlk_status_string(0).decode() == "ok"
    assert "workspace" in lib.rlk_status_string(3).decode()


def test_workspace_queries(lib):
    # forward: three fp32 arrays of ceil(V_local/1024) x T, each rounded up to 256 bytes,
    # then 256 bytes of work-item counters
    T, V = 4096, 151936
    per = -(-(V // 1024 + (V % 1024 > 0)) * T * 4 // 256) * 256
    assert lib.rlk_linear_logp_fwd_workspace(T, 4096, V) == 3 * per + 256
    # backward: bf16 dz tiles [T][round_up(V_local, 256)] + fp32 [T][H] running sum of dH
    # + the counters
    assert lib.rlk_linear_logp_bwd_workspace(T, 4096, V) == T * 152064 * 2 + T * 4096 * 4 + 256
    assert lib.rlk_linear_logp_bwd_workspace(T, 4096, 16384) == T * 16384 * 2 + 256  # one chunk
    assert lib.rlk_linear_logp_fwd_workspace(0, 4096, V) == 0
    assert lib.rlk_linear_logp_bwd_workspace(0, 4096, V) == 0


def fwd(lib, h=FAKE, W=FAKE, y=FAKE, T=4, H=64, V_local=4096, vocab_start=0, V_true=4096,
        logp=FAKE, lse=FAKE, partial=None, ws=FAKE, ws_bytes=1 << 30):
    return lib.rlk_linear_logp_fwd(h, W, y, T, H, V_local, vocab_start, V_true, logp, lse, partial,
                                   None, ws, ws_bytes, None)


def bwd(lib, h=FAKE, W=FAKE, y=FAKE, lse=FAKE, g=FAKE, T=4, H=64, V_local=4096, vocab_start=0,
        V_true=4096, dH=FAKE, dW=FAKE, ws=FAKE, ws_bytes=1 << 30):
    return lib.rlk_linear_logp_bwd(h, W, y, lse, g, T, H, V_local, vocab_start, V_true, dH, 0, dW,
                                   None, ws, ws_bytes, None)


def test_forward_argument_errors(lib):
    assert fwd(lib, h=None) == INVALID
    assert fwd(lib, W=None) == INVALID
    assert fwd(lib, y=None) == INVALID
    assert fwd(lib, T=-1) == INVALID
    assert fwd(lib, H=60) == INVALID            # H % 8 != 0
    assert fwd(lib, h=MISALIGNED) == INVALID
    assert fwd(lib, V_true=0) == INVALID
    assert fwd(lib, logp=None, lse=None) == INVALID
    assert fwd(lib, V_true=1 << 25, V_local=1 << 25) == UNSUPPORTED
    # unsharded output needs the whole [0, V_true)
    assert fwd(lib, T=0, V_local=2048, V_true=4096) == INVALID


def test_forward_empty_and_workspace(lib):
    assert fwd(lib, T=0) == OK
    assert fwd(lib, T=0, h=None, y=None) == OK        # an empty batch has no storage
    assert fwd(lib, T=0, h=None, y=None, logp=None, lse=None) == OK
    assert fwd(lib, T=0, W=None) == INVALID
    assert fwd(lib, T=0, h=FAKE, ws=None, ws_bytes=0) == OK
    need = lib.rlk_linear_logp_fwd_workspace(4, 64, 4096)
    assert fwd(lib, ws_bytes=need - 1) == WORKSPACE
    assert fwd(lib, ws=None) == WORKSPACE
    assert fwd(lib, ws=ctypes.c_void_p(0x100010)) == WORKSPACE   # not 256-byte aligned


def test_shard_splits_the_tree_accepts(lib):
    import deterministic_token_logprob_gb300 as rlk
    V, Vt = 151936, 151669
    for S in (1, 2, 4, 8):
        for start, vl in rlk.shard_bounds(V, Vt, S):
            assert fwd(lib, T=0, V_local=vl, vocab_start=start, V_true=Vt, logp=None, lse=None,
                       partial=FAKE) == OK, (S, start, vl)
    # the split used by the Qwen3-30B-A3B workload: super-shard width 19 * 1024
    assert rlk.shard_bounds(V, Vt, 2) == [(0, 77824), (77824, 74112)]


def test_shard_splits_the_tree_rejects(lib):
    V, Vt = 151936, 151669
    P = dict(T=0, V_true=Vt, logp=None, lse=None, partial=FAKE)
    assert fwd(lib, V_local=75968, vocab_start=75968, **P) == UNSUPPORTED   # equal halves: not tree-aligned
    assert fwd(lib, V_local=75968, vocab_start=0, **P) == UNSUPPORTED
    assert fwd(lib, V_local=3 * 19456, vocab_start=0, **P) == UNSUPPORTED   # 3 super-shards
    assert fwd(lib, V_local=2 * 19456, vocab_start=19456, **P) == UNSUPPORTED  # misaligned pair
    assert fwd(lib, V_local=19456, vocab_start=19456 * 8, **P) == UNSUPPORTED  # beyond the tree


def test_backward_argument_errors(lib):
    assert bwd(lib, lse=None) == INVALID
    assert bwd(lib, g=None) == INVALID
    assert bwd(lib, dW=MISALIGNED) == INVALID
    assert bwd(lib, H=12) == INVALID
    assert bwd(lib, T=0) == OK
    assert bwd(lib, T=0, h=None, y=None, lse=None, g=None, dH=None, dW=None) == OK
    need = lib.rlk_linear_logp_bwd_workspace(4, 64, 4096)
    assert bwd(lib, ws_bytes=need - 1) == WORKSPACE
    assert bwd(lib, ws=None) == WORKSPACE


def test_backward_stages_argument_errors(lib):
    def st(stages, dH=FAKE, dW=FAKE, T=4, ws_bytes=1 << 30):
        return lib.rlk_linear_logp_bwd_stages(FAKE, FAKE, FAKE, FAKE, FAKE, T, 64, 4096, 0, 4096, dH,
                                              0, dW, stages, None, FAKE, ws_bytes, None)
    DZ, DH, DW = 1, 2, 4
    assert st(0) == INVALID                   # no stage
    assert st(8) == INVALID                   # unknown bit
    assert st(DZ | 16) == INVALID
    assert st(DH, dH=None) == INVALID         # a selected output may not be missing
    assert st(DW, dW=None) == INVALID
    assert st(DZ | DH | DW, dH=None) == INVALID
    assert st(DZ, dH=None, dW=None, T=0) == OK
    assert st(DH, T=0) == OK
    need = lib.rlk_linear_logp_bwd_workspace(4, 64, 4096)
    assert st(DZ, ws_bytes=need - 1) == WORKSPACE
    assert st(DW, ws_bytes=need - 1) == WORKSPACE


def test_merge_and_sum_argument_errors(lib):
    assert lib.rlk_lse_merge(FAKE, 3, 10, FAKE, FAKE, None) == UNSUPPORTED
    assert lib.rlk_lse_merge(None, 2, 10, FAKE, FAKE, None) == INVALID
    assert lib.rlk_lse_merge(FAKE, 2, 0, FAKE, FAKE, None) == OK
    assert lib.rlk_lse_merge(None, 2, 0, None, None, None) == OK
    assert lib.rlk_shard_sum_bf16(FAKE, 2, 0, FAKE, None) == OK
    assert lib.rlk_shard_sum_bf16(MISALIGNED, 2, 8, FAKE, None) == INVALID
    assert lib.rlk_shard_sum_bf16(FAKE, 0, 8, FAKE, None) == INVALID


def test_saved_logits_queries_and_errors(lib):
    assert lib.rlk_saved_logits_bytes(8192, 151936) == 8192 * 152064 * 4
    assert lib.rlk_saved_logits_bytes(0, 151936) == 0
    need = lib.rlk_saved_logits_bytes(4, 4096)
    args = (FAKE, FAKE, FAKE, 4, 64, 4096, 0, 4096, FAKE, FAKE, None)
    assert lib.rlk_linear_logp_fwd_save(*args, None, need, None, FAKE, 1 << 30, None) == INVALID
    assert lib.rlk_linear_logp_fwd_save(*args, FAKE, need - 1, None, FAKE, 1 << 30, None) == INVALID
    assert lib.rlk_linear_logp_fwd_save(*args, MISALIGNED, need, None, FAKE, 1 << 30, None) == INVALID
    bargs = (FAKE, FAKE, FAKE, FAKE, FAKE)
    rest = (4, 64, 4096, 0, 4096, FAKE, 0, FAKE, None, FAKE, 1 << 30, None)
    assert lib.rlk_linear_logp_bwd_saved(*bargs, None, need, *rest) == INVALID
    assert lib.rlk_linear_logp_bwd_saved(*bargs, FAKE, need - 1, *rest) == INVALID
    zero = (0, 64, 4096, 0, 4096, None, 0, None, None, None, 0, None)
    assert lib.rlk_linear_logp_bwd_saved(None, FAKE, None, None, None, None, 0, *zero) == OK


def test_saved_probs_queries_and_errors(lib):
    T, V = 8192, 151936
    Vd = 152064
    assert lib.rlk_saved_probs_bytes(T, V) == -(-T * Vd * 2 // 256) * 256 + T * (Vd // 64) * 4
    need = lib.rlk_saved_probs_bytes(4, 4096)
    args = (FAKE, FAKE, FAKE, 4, 64, 4096, 0, 4096, FAKE, FAKE, None)
    assert lib.rlk_linear_logp_fwd_save_probs(*args, None, need, None, FAKE, 1 << 30, None) == INVALID
    assert lib.rlk_linear_logp_fwd_save_probs(*args, FAKE, need - 1, None, FAKE, 1 << 30, None) == INVALID
    assert lib.rlk_linear_logp_fwd_save_probs(*args, ctypes.c_void_p(0x100010), need, None, FAKE,
                                              1 << 30, None) == INVALID      # not 256-aligned
    bargs = (FAKE, FAKE, FAKE, FAKE, FAKE)
    rest = (4, 64, 4096, 0, 4096, FAKE, 0, FAKE, None, FAKE, 1 << 30, None)
    assert lib.rlk_linear_logp_bwd_saved_probs(*bargs, None, need, *rest) == INVALID
    assert lib.rlk_linear_logp_bwd_saved_probs(*bargs, FAKE, need - 1, *rest) == INVALID


def test_fp8_argument_errors(lib):
    # quantizer
    assert lib.rlk_quantize_rows_e4m3(FAKE, 0, 64, FAKE, FAKE, None, None) == OK
    assert lib.rlk_quantize_rows_e4m3(None, 0, 0, None, None, None, None) == OK
    assert lib.rlk_quantize_rows_e4m3(FAKE, -1, 64, FAKE, FAKE, None, None) == INVALID
    assert lib.rlk_quantize_rows_e4m3(FAKE, 4, 60, FAKE, FAKE, None, None) == INVALID  # cols % 8
    assert lib.rlk_quantize_rows_e4m3(MISALIGNED, 4, 64, FAKE, FAKE, None, None) == INVALID
    assert lib.rlk_quantize_rows_e4m3(FAKE, 4, 64, FAKE, None, None, None) == INVALID
    # forward: hq, h_scale, Wq, W_scale, y, T, H, V_local, vocab_start, V_true, logp, lse, partial,
    #          err, ws, ws_bytes, stream
    ws = lib.rlk_linear_logp_fwd_workspace(4, 64, 4096)

    def f8(**k):
        a = dict(hq=FAKE, hs=FAKE, Wq=FAKE, Ws=FAKE, y=FAKE, T=4, H=64, V=4096, vs=0, Vt=4096,
                 logp=FAKE, lse=FAKE, part=None, err=None, ws=FAKE, nb=ws, s=None)
        a.update(k)
        return lib.rlk_linear_logp_fwd_fp8(*a.values())

    assert f8(T=0) == OK
    assert f8(H=72) == INVALID                 # H % 16 != 0 (E4M3 rows need 16-byte strides)
    assert f8(hs=None) == INVALID
    assert f8(Ws=None) == INVALID
    assert f8(Ws=ctypes.c_void_p(0x100004)) == INVALID   # W_scale not 16-byte aligned
    assert f8(Wq=MISALIGNED) == INVALID
    assert f8(nb=ws - 1) == WORKSPACE
    assert f8(T=0, hq=None, hs=None, y=None) == OK
    # backward: h, W, hq, h_scale, Wq, W_scale, y, lse, g, T, H, V_local, vocab_start, V_true,
    #           dH, partial, dW, err, ws, ws_bytes, stream
    bws = lib.rlk_linear_logp_bwd_workspace(4, 64, 4096)

    def b8(**k):
        a = dict(h=FAKE, W=FAKE, hq=FAKE, hs=FAKE, Wq=FAKE, Ws=FAKE, y=FAKE, lse=FAKE, g=FAKE, T=4,
                 H=64, V=4096, vs=0, Vt=4096, dH=FAKE, part=0, dW=FAKE, err=None, ws=FAKE, nb=bws,
                 s=None)
        a.update(k)
        return lib.rlk_linear_logp_bwd_fp8(*a.values())

    assert b8(T=0) == OK
    assert b8(Wq=None) == INVALID
    assert b8(hq=MISALIGNED) == INVALID
    assert b8(H=72) == INVALID
    assert b8(Ws=None) == INVALID
    assert b8(nb=bws - 1) == WORKSPACE


def test_debug_checks_variant_builds_and_exports_the_same_symbols(lib):
    # the variant with device-side index checks (compiled here, run by the GPU tests)
    import subprocess
    from deterministic_token_logprob_gb300 import _binding, build
    path = build.build(debug_checks=True)
    assert path != build.LIB

    def exported(p):
        out = subprocess.run(["nm", "-D", "--defined-only", p], capture_output=True, text=True).stdout
        return {ln.split()[-1] for ln in out.splitlines() if " T " in ln and ln.split()[-1].startswith("rlk_")}
    assert exported(path) == exported(build.LIB) == set(declared_functions())
    dbg = _binding._declare(ctypes.CDLL(path))
    assert dbg.rlk_debug_checks() == 1
    assert lib.rlk_debug_checks() == 0
    # without the checks the bounds self-test is refused before anything touches CUDA
    args = (FAKE, FAKE, FAKE, 4, 64, 4096, 4096, FAKE, FAKE, FAKE, FAKE, 1 << 30, None)
    assert lib.rlk_selftest_bounds_check(*args) == UNSUPPORTED
    assert dbg.rlk_selftest_bounds_check(FAKE, FAKE, FAKE, 4, 64, 4096, 4096, FAKE, FAKE, None, FAKE,
                                         1 << 30, None) == INVALID   # err_flag is required
