"""The C-ABI library: it builds, loads, exports every declared entry point, and rejects
bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dgsamp.h")


@pytest.fixture(scope="module")
def lib():
    from denoising_sampler_step_gb300 import build
    build.build()
    from denoising_sampler_step_gb300 import binding
    return binding


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dg_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ["dg_row_stats", "dg_soft_embed", "dg_entropy_accept", "dg_sum_partials", "dg_sampler_step",
              "dg_soft_embed_workspace_size", "dg_get_device_status", "dg_last_error", "dg_version",
              "dg_row_sample", "dg_entropy_accept_eligible", "dg_loop_update", "dg_sampler_loop_step",
              "dg_row_stats_sample", "dg_row_stats_partial", "dg_row_stats_combine"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for n in declared_symbols():
        assert hasattr(so, n), n


def test_python_binding_names_match_c(lib):
    for n in declared_symbols():
        if n in ("dg_last_error", "dg_version"):
            continue
        assert callable(getattr(lib, n)), n


def test_version(lib):
    assert lib.lib.dg_version() == 100


def test_row_stats_rejects_bad_arguments(lib):
    L = lib.lib
    assert L.dg_row_stats(None, 4, 16, 16, None, None, None, None, None, None) == 1
    assert L.dg_row_stats(ctypes.c_void_p(16), 4, 0, 16, None, None, None, None, None, None) == 1
    assert L.dg_row_stats(ctypes.c_void_p(16), 4, 32, 16, None, None, None, None, None, None) == 1
    # misaligned base or leading dimension
    assert L.dg_row_stats(ctypes.c_void_p(20), 4, 16, 16, None, None, None, None, None, None) == 2
    assert L.dg_row_stats(ctypes.c_void_p(16), 4, 15, 15, None, None, None, None, None, None) == 2
    assert b"16-byte" in L.dg_last_error()
    # nothing to do: no launch, no error
    assert L.dg_row_stats(None, 0, 16, 16, None, None, None, None, None, None) == 0


def test_accept_rejects_bad_arguments(lib):
    L = lib.lib
    p = ctypes.c_void_p(256)
    assert L.dg_entropy_accept(p, p, 1, 1025, p, 0, p, p, p, None) == 2
    assert L.dg_entropy_accept(p, p, 1, 0, p, 0, p, p, p, None) == 1
    assert L.dg_entropy_accept(p, p, -1, 16, p, 0, p, p, p, None) == 1
    assert L.dg_entropy_accept(p, p, 1, 16, p, -1, p, p, p, None) == 1
    assert L.dg_entropy_accept(None, p, 1, 16, p, 0, p, p, p, None) == 1
    assert L.dg_entropy_accept(None, None, 0, 16, None, 0, None, None, None, None) == 0


def test_soft_embed_rejects_the_contraction_mismatch(lib):
    """The pages' crash: a slice of e-s vocabulary entries against a shard with fewer
    rows.  The library answers with an error instead of reading out of range."""
    L = lib.lib
    p = ctypes.c_void_p(256)
    # 262144 probabilities against a 65536-row shard
    st = L.dg_soft_embed(p, 262144, p, 256, 0, 262144, p, 65536, 2816, 2816, 53.0, p, 2816, p, 1 << 30, None)
    assert st == 1 and b"shard" in L.dg_last_error()
    assert L.dg_soft_embed(p, 4096, p, 16, 100, 50, p, 4096, 256, 256, 1.0, p, 256, p, 1 << 20, None) == 1
    assert L.dg_soft_embed(p, 4096, p, 16, 0, 5000, p, 8192, 256, 256, 1.0, p, 256, p, 1 << 20, None) == 1
    assert L.dg_soft_embed(p, 4096, p, 16, 0, 4096, p, 4096, 100, 256, 1.0, p, 256, p, 1 << 20, None) == 1
    # unaligned W leading dimension / logits leading dimension
    assert L.dg_soft_embed(p, 4096, p, 16, 0, 4096, p, 4096, 260, 258, 1.0, p, 258, p, 1 << 20, None) == 2
    assert L.dg_soft_embed(p, 4097, p, 16, 0, 4096, p, 4096, 256, 256, 1.0, p, 256, p, 1 << 20, None) == 2


def test_sum_partials_rejects_bad_arguments(lib):
    L = lib.lib
    arr = (ctypes.c_void_p * 17)(*([256] * 17))
    assert L.dg_sum_partials(arr, 0, 4, 4, 4, 1.0, ctypes.c_void_p(256), 4, None) == 1
    assert L.dg_sum_partials(arr, 17, 4, 4, 4, 1.0, ctypes.c_void_p(256), 4, None) == 1
    arr2 = (ctypes.c_void_p * 2)(256, None)
    assert L.dg_sum_partials(arr2, 2, 4, 4, 4, 1.0, ctypes.c_void_p(256), 4, None) == 1


def test_row_sample_rejects_bad_temperatures(lib):
    L = lib.lib
    p = ctypes.c_void_p(256)
    for t in (0.0, -1.0, float("inf"), float("nan")):
        assert L.dg_row_sample(p, 4, 16, 16, t, 1, 0, p, p, None) == 1, t
    assert b"temperature" in L.dg_last_error()
    assert L.dg_row_sample(p, 4, 16, 18, 1.0, 1, 0, p, p, None) == 2  # ldl % 4 != 0


def test_wait_timeout_check_rejects_bad_limits(lib):
    L = lib.lib
    assert L.dg_check_wait_timeout(0, None) == 1
    assert b"outside" in L.dg_last_error()
    assert L.dg_check_wait_timeout(1000001, None) == 1


def test_step_checks_slice_against_vocabulary(lib):
    L = lib.lib
    p = ctypes.c_void_p(256)
    st = L.dg_sampler_step(p, 1, 16, 4096, 4096, p, 0, 8192, 8192, 256, 256, 16.0, p, 0,
                           p, p, p, p, p, p, p, p, p, 256, 0, p, 1 << 20, None)
    assert st == 1


def test_step_rejects_unknown_flags(lib):
    L = lib.lib
    p = ctypes.c_void_p(256)
    for flags in (2, 1 << 31, 3):
        st = L.dg_sampler_step(p, 1, 16, 4096, 4096, p, 0, 4096, 4096, 256, 256, 16.0, p, 0,
                               p, p, p, p, p, p, p, p, p, 256, flags, p, 1 << 20, None)
        assert st == 1 and b"flags" in L.dg_last_error(), flags
        st = L.dg_sampler_step_e4m3(p, 1, 16, 4096, 4096, p, p, 0, 4096, 4096, 256, 256, 1.0, p, 0, p, p, p, p, p,
                                    p, p, p, p, 256, flags, p, 1 << 20, None)
        assert st == 1 and b"flags" in L.dg_last_error(), flags
    assert lib.DG_STEP_TWO_PASS == 1


def test_accept_eligible_rejects_bad_arguments(lib):
    L = lib.lib
    p = ctypes.c_void_p(256)
    assert L.dg_entropy_accept_eligible(p, p, None, 1, 16, p, 0, p, p, p, None) == 1
    assert b"eligible" in L.dg_last_error()
    assert L.dg_entropy_accept_eligible(p, p, p, 1, 1025, p, 0, p, p, p, None) == 2
    assert L.dg_entropy_accept_eligible(p, p, p, 1, 16, p, -1, p, p, p, None) == 1
    assert L.dg_entropy_accept_eligible(None, None, None, 0, 16, None, 0, None, None, None, None) == 0


def test_loop_update_rejects_bad_arguments(lib):
    L = lib.lib
    p = ctypes.c_void_p(256)
    state = [p] * 6
    assert L.dg_loop_update(p, p, p, p, -1, 16, 2, 0.5, 10, *state, None) == 1
    assert L.dg_loop_update(p, p, p, p, 1, 0, 2, 0.5, 10, *state, None) == 1
    assert L.dg_loop_update(p, p, p, p, 1, 1025, 2, 0.5, 10, *state, None) == 2
    assert L.dg_loop_update(p, p, p, p, 1, 16, -1, 0.5, 10, *state, None) == 1
    assert L.dg_loop_update(p, p, p, p, 1, 16, 2, 0.5, 0, *state, None) == 1
    assert L.dg_loop_update(p, p, p, p, 1, 16, 2, float("nan"), 10, *state, None) == 1
    assert L.dg_loop_update(p, p, p, p, 1, 16, 2, 0.5, 10, p, p, None, p, p, p, None) == 1
    assert L.dg_loop_update(None, p, p, p, 1, 16, 2, 0.5, 10, *state, None) == 1
    assert L.dg_loop_update(p, None, p, p, 1, 16, 2, 0.5, 10, *state, None) == 1
    assert L.dg_loop_update(None, None, None, None, 0, 16, 2, 0.5, 10, *([None] * 6), None) == 0


def test_loop_step_checks_its_loop_arguments(lib):
    L = lib.lib
    p = ctypes.c_void_p(256)
    step = [p, 1, 16, 4096, 4096, p, 0, 4096, 4096, 256, 256, 16.0, p, 0]
    outs = [p] * 10 + [256]
    ws = [0, p, 1 << 20, None]   # flags, workspace, its size, stream
    argmax_mode = [0.0, 0, 0]
    assert L.dg_sampler_loop_step(*step, 2, 0.5, 0, *argmax_mode, *outs, *([p] * 6), *ws) == 1   # step_limit 0
    assert L.dg_sampler_loop_step(*step, 2, 0.5, 10, *argmax_mode, *outs, p, None, p, p, p, p, *ws) == 1
    bad = list(step)
    bad[7] = 8192                                                                              # slice past V
    assert L.dg_sampler_loop_step(*bad, 2, 0.5, 10, *argmax_mode, *outs, *([p] * 6), *ws) == 1
    for t in (-1.0, float("inf"), float("nan")):
        assert L.dg_sampler_loop_step(*step, 2, 0.5, 10, t, 1, 0, *outs, *([p] * 6), *ws) == 1, t
    no_cand = [p] * 5 + [None] + [p] * 4 + [256]                                               # candidate NULL
    assert L.dg_sampler_loop_step(*step, 2, 0.5, 10, 1.0, 1, 0, *no_cand, *([p] * 6), *ws) == 1
    assert b"candidate" in L.dg_last_error()


def test_row_stats_sample_rejects_bad_arguments(lib):
    L = lib.lib
    p = ctypes.c_void_p(256)
    for t in (0.0, -1.0, float("inf"), float("nan")):
        assert L.dg_row_stats_sample(p, 4, 16, 16, t, 1, 0, p, p, p, p, p, p, p, None) == 1, t
    assert L.dg_row_stats_sample(p, 4, 16, 16, 1.0, 1, 0, p, p, p, p, p, None, p, None) == 1
    assert L.dg_row_stats_sample(p, 4, 16, 18, 1.0, 1, 0, p, p, p, p, p, p, p, None) == 2  # ldl % 4 != 0
    assert L.dg_row_stats_sample(None, 0, 16, 16, 1.0, 1, 0, *([None] * 7), None) == 0


def test_sharded_statistics_reject_bad_arguments(lib):
    L = lib.lib
    p = ctypes.c_void_p(256)
    assert L.dg_row_stats_partial(p, 4, 16, 16, -1, p, None) == 1            # negative offset
    assert L.dg_row_stats_partial(p, 4, 16, 16, 2**31 - 10, p, None) == 1    # past int32 indices
    assert L.dg_row_stats_partial(p, 4, 16, 16, 0, None, None) == 1
    assert L.dg_row_stats_partial(p, 4, 16, 16, 0, ctypes.c_void_p(264), None) == 2   # state not 16-byte aligned
    assert L.dg_row_stats_partial(p, 4, 16, 18, 0, p, None) == 2             # ldl % 4 != 0
    assert L.dg_row_stats_combine(p, 0, 4, p, p, p, p, p, None) == 1
    assert L.dg_row_stats_combine(p, 1025, 4, p, p, p, p, p, None) == 1
    assert L.dg_row_stats_combine(None, 2, 4, p, p, p, p, p, None) == 1
    assert L.dg_row_stats_combine(ctypes.c_void_p(264), 2, 4, p, p, p, p, p, None) == 2
    assert L.dg_row_stats_combine(None, 2, 0, None, None, None, None, None, None) == 0


def test_e4m3_calls_reject_bad_arguments(lib):
    L = lib.lib
    p = ctypes.c_void_p(256)
    # quantiser: sizes, NULL pointers, alignment
    assert L.dg_quantize_e4m3(p, 4, 0, 16, p, 16, p, None) == 1
    assert L.dg_quantize_e4m3(p, 4, 32, 16, p, 32, p, None) == 1
    assert L.dg_quantize_e4m3(None, 4, 16, 16, p, 16, p, None) == 1
    assert L.dg_quantize_e4m3(ctypes.c_void_p(258), 4, 16, 16, p, 16, p, None) == 2
    assert L.dg_quantize_e4m3(p, 4, 15, 15, p, 16, p, None) == 2
    assert L.dg_quantize_e4m3(None, 0, 16, 16, None, 16, None, None) == 0
    # product: the contraction mismatch, a missing scale array, unaligned codes
    st = L.dg_soft_embed_e4m3(p, 262144, p, 256, 0, 262144, p, p, 65536, 2816, 2816, 53.0, p, 2816, p, 1 << 30, None)
    assert st == 1 and b"shard" in L.dg_last_error()
    assert L.dg_soft_embed_e4m3(p, 4096, p, 16, 0, 4096, p, None, 4096, 256, 256, 1.0, p, 256, p, 1 << 20, None) == 1
    assert L.dg_soft_embed_e4m3(p, 4096, p, 16, 0, 4096, p, p, 4096, 264, 260, 1.0, p, 260, p, 1 << 20, None) == 2
    assert L.dg_soft_embed_e4m3(p, 4096, p, 16, 0, 4096, ctypes.c_void_p(264), p, 4096, 256, 256, 1.0, p, 256, p,
                                1 << 20, None) == 2
    assert L.dg_soft_embed_e4m3(p, 4096, p, 16, 0, 4096, p, ctypes.c_void_p(258), 4096, 256, 256, 1.0, p, 256, p,
                                1 << 20, None) == 2
    # the step checks its slice against V like the bf16 step
    st = L.dg_sampler_step_e4m3(p, 1, 16, 4096, 4096, p, p, 0, 5000, 8192, 256, 256, 1.0, p, 0, p, p, p, p, p, p, p,
                                p, p, 256, 0, p, 1 << 20, None)
    assert st == 1
