"""The C ABI library: it loads, exports every function include/td.h declares, and rejects
bad arguments on the host before launching anything (CPU, no GPU needed)."""

import ctypes
import os
import re

import pytest
import torch

import block_diffusion_lm_denoise_b300 as td

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    src = open(os.path.join(ROOT, "include", "td.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(td_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(td.LIB_PATH):
        from block_diffusion_lm_denoise_b300 import build
        build.build()
    return td.lib()


def test_every_declared_function_is_exported(lib):
    declared = _header_functions()
    assert set(declared) == set(td.EXPORTED), declared
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in enumerate(["TD_OK", "TD_ERR_INVALID_ARG", "TD_ERR_WORKSPACE",
                                 "TD_ERR_UNSUPPORTED", "TD_ERR_CUDA", "TD_ERR_NOT_CONVERGED",
                                 "TD_ERR_DEVICE_TIMEOUT"]):
        assert lib.td_status_string(code).decode() == name


def test_workspace_sizes_and_unsupported_shapes(lib):
    ok = td.make_dims(B=64, S=16, d=4096, Hq=32, Hkv=2, D=128, V=131072, Lmax=8192, n_layers=6)
    for fn in (td.TD_FN_BLOCK_ATTENTION, td.TD_FN_LMHEAD_COMMIT, td.TD_FN_DENOISE_STEP,
               td.TD_FN_DECODE_BLOCK):
        assert td.td_workspace_size(ok, fn) > 0
    assert td.td_workspace_size(ok, td.TD_FN_ADALN_MODULATE) == 0
    for bad in (dict(D=96), dict(Hq=30, Hkv=4), dict(S=65), dict(d=100)):
        dm = td.make_dims(**{**dict(B=2, S=16, d=256, Hq=4, Hkv=1, D=64, V=1024, Lmax=64,
                                     n_layers=1), **bad})
        with pytest.raises(td.TdError):
            td.td_workspace_size(dm, td.TD_FN_DENOISE_STEP)


def test_null_pointers_are_rejected_before_any_launch(lib):
    dm = td.make_dims(B=1, S=16, d=256, Hq=4, Hkv=1, D=64, V=1024, Lmax=64, n_layers=1)
    # every pointer null: validation must fail first
    assert lib.td_block_attention(ctypes.byref(dm), None, None, None, None, None, None, None, 0,
                                  None, None, None, 0, None) == 1
    assert lib.td_lmhead_commit(ctypes.byref(dm), None, None, 0.8, 0, 0, None, None, None, None,
                                None, None, None, 0, None) == 1
    assert lib.td_adaln_modulate(None, None, None, 4, 256, 1e-6, None, None) == 1
    steps = ctypes.c_int(0)
    assert lib.td_decode_block(ctypes.byref(dm), None, None, None, None, None, None, 1, 16,
                               0.8, None, None, None, None, None, None, None, ctypes.byref(steps),
                               None, 0, None) == 1
    assert lib.td_kv_append(ctypes.byref(dm), None, None, None, None, None) == 1
    # shapes outside the kernels' limits
    bad = td.make_dims(B=1, S=16, d=256, Hq=4, Hkv=1, D=80, V=1024, Lmax=64, n_layers=1)
    fake = ctypes.c_void_p(1 << 40)   # never dereferenced: the shape check fails first
    assert lib.td_block_attention(ctypes.byref(bad), fake, fake, fake, fake, fake, None, None, 0,
                                  fake, None, fake, 1 << 20, None) == 3


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake device pointers only without a GPU")
def test_undersized_workspace_is_rejected(lib):
    dm = td.make_dims(B=1, S=16, d=256, Hq=4, Hkv=1, D=64, V=1024, Lmax=64, n_layers=1)
    fake = ctypes.c_void_p(1 << 40)
    assert lib.td_block_attention(ctypes.byref(dm), fake, fake, fake, fake, fake, None, None, 0,
                                  fake, None, fake, 16, None) == 2


def test_unknown_commit_rule_is_rejected(lib):
    dm = td.make_dims(B=1, S=16, d=256, Hq=4, Hkv=1, D=64, V=1024, Lmax=64, n_layers=1)
    fake = ctypes.c_void_p(1 << 40)   # never dereferenced: the rule check fails first
    assert lib.td_lmhead_commit(ctypes.byref(dm), fake, fake, 0.8, 7, 0, fake, fake, fake, fake,
                                fake, fake, fake, 1 << 30, None) == 1


def test_invalid_step_options_are_rejected(lib):
    dm = td.make_dims(B=1, S=16, d=256, Hq=4, Hkv=1, D=64, V=1024, Lmax=64, n_layers=0)
    fake = ctypes.c_void_p(1 << 40)   # never dereferenced: the option check fails first
    steps = ctypes.c_int(0)
    for opts in (td.td_step_opts(5, 0.0), td.td_step_opts(0, -1.0),
                 td.td_step_opts(0, float("nan")),
                 td.td_step_opts(0, 0.0, td.td_paging(), None, 2)):   # unknown precision
        assert lib.td_denoise_step(ctypes.byref(dm), None, None, fake, fake, fake, fake, fake, 1,
                                   16, 0.8, ctypes.byref(opts), fake, fake, fake, fake, fake,
                                   fake, fake, 1 << 30, None) == 1
        assert lib.td_decode_block(ctypes.byref(dm), None, None, fake, fake, fake, fake, 1, 16,
                                   0.8, ctypes.byref(opts), fake, fake, fake, fake, fake, fake,
                                   ctypes.byref(steps), fake, 1 << 30, None) == 1


def test_malformed_paging_is_rejected(lib):
    dm = td.make_dims(B=2, S=16, d=256, Hq=4, Hkv=1, D=64, V=1024, Lmax=300, n_layers=1)
    fake = ctypes.c_void_p(1 << 40)   # never dereferenced: the paging check fails first
    for pg in (td.td_paging(fake, 2, 8),     # 2 columns cannot cover Lmax = 300 (3 tiles)
               td.td_paging(fake, 3, 0)):    # empty pool
        assert lib.td_block_attention(ctypes.byref(dm), fake, fake, fake, fake, fake, None,
                                      ctypes.byref(pg), 0, fake, None, fake, 1 << 30,
                                      None) == 1
        assert lib.td_kv_append(ctypes.byref(dm), None, None, fake, ctypes.byref(pg), None) == 1


def test_adaln_shape_and_alignment_checks(lib):
    fake = ctypes.c_void_p(1 << 40)        # never dereferenced: the checks fail first
    odd = ctypes.c_void_p((1 << 40) + 2)   # bf16-aligned but off a 16-byte boundary
    assert lib.td_adaln_modulate(fake, fake, fake, 4, 8200, 1e-6, fake, None) == 3   # d > 8192
    assert lib.td_adaln_modulate(fake, fake, fake, 4, 260, 1e-6, fake, None) == 3    # d % 8
    assert lib.td_adaln_modulate(odd, fake, fake, 4, 256, 1e-6, fake, None) == 1
    assert lib.td_adaln_modulate(fake, fake, fake, 4, 256, 1e-6, odd, None) == 1
    assert lib.td_adaln_modulate(fake, fake, fake, 4, 256, -1.0, fake, None) == 1     # eps < 0


def test_step_and_loop_reject_misaligned_tables_before_any_launch(lib):
    dm = td.make_dims(B=1, S=16, d=256, Hq=4, Hkv=1, D=64, V=1024, Lmax=0, n_layers=0)
    fake = ctypes.c_void_p(1 << 40)        # never dereferenced: the checks fail first
    odd = ctypes.c_void_p((1 << 40) + 2)   # bf16-aligned but off a 16-byte boundary
    steps = ctypes.c_int(0)
    for emb, pos, w in ((odd, fake, fake), (fake, odd, fake), (fake, fake, odd)):
        # embedding path (h = NULL)
        assert lib.td_denoise_step(ctypes.byref(dm), None, None, None, emb, pos, w, fake, 1,
                                   16, 0.8, None, fake, fake, fake, fake, fake, fake, fake,
                                   1 << 30, None) == 1
        assert lib.td_decode_block(ctypes.byref(dm), None, None, emb, pos, w, fake, 1, 16,
                                   0.8, None, fake, fake, fake, fake, fake, fake,
                                   ctypes.byref(steps), fake, 1 << 30, None) == 1
    # with h given, emb / pos are not read and may be anything; w_lm still must be aligned
    assert lib.td_denoise_step(ctypes.byref(dm), None, None, odd, None, None, odd, fake, 1, 16,
                               0.8, None, fake, fake, fake, fake, fake, fake, fake, 1 << 30,
                               None) == 1


def test_static_entry_point_rejects_sizes_beyond_its_scratch_before_any_cuda_call(lib):
    # 16 MiB of scratch holds the LM-head partials of B*S <= 2048 rows at V = 131072
    # (12 bytes per row and 256-wide vocabulary tile); beyond that: TD_ERR_WORKSPACE
    fake = ctypes.c_void_p(1 << 40)        # never dereferenced: the size check fails first
    big = td.make_dims(B=256, S=16, d=4096, Hq=32, Hkv=2, D=128, V=131072, Lmax=0, n_layers=0)
    assert lib.td_lmhead_commit_static(ctypes.byref(big), fake, fake, 0.8, 0, fake, fake, fake,
                                       fake, fake, fake, None) == 2
    odd = ctypes.c_void_p((1 << 40) + 2)
    ok = td.make_dims(B=64, S=16, d=4096, Hq=32, Hkv=2, D=128, V=131072, Lmax=0, n_layers=0)
    assert lib.td_lmhead_commit_static(ctypes.byref(ok), odd, fake, 0.8, 0, fake, fake, fake,
                                       fake, fake, fake, None) == 1


def test_workspace_sizes_grow_with_the_problem():
    base = dict(B=8, S=16, d=4096, Hq=32, Hkv=2, D=128, V=131072, Lmax=2048, n_layers=2)

    def ws(fn, **kw):
        return td.td_workspace_size(td.make_dims(**{**base, **kw}), fn)

    for fn in (td.TD_FN_BLOCK_ATTENTION, td.TD_FN_LMHEAD_COMMIT, td.TD_FN_DENOISE_STEP):
        assert ws(fn, B=16) >= ws(fn, B=8)
    assert ws(td.TD_FN_LMHEAD_COMMIT, V=262144) > ws(td.TD_FN_LMHEAD_COMMIT)
    # a step holds the attention's and the LM head's scratch besides its activations
    step = ws(td.TD_FN_DENOISE_STEP)
    assert step >= ws(td.TD_FN_LMHEAD_COMMIT) and step >= ws(td.TD_FN_BLOCK_ATTENTION)
    # the loop runs the step: the same workspace
    assert ws(td.TD_FN_DECODE_BLOCK) == step


def test_timestep_table_validates_on_the_host(lib):
    p = ctypes.c_void_p(16)   # never dereferenced: every call below is rejected first
    assert lib.td_timestep_table(None, p, 64, 16, p, None) == 1
    assert lib.td_timestep_table(p, p, 0, 16, p, None) == 1
    assert lib.td_timestep_table(p, p, 64, 0, p, None) == 1
    assert lib.td_timestep_table(p, p, 64, 65537, p, None) == 1
    assert lib.td_timestep_table(p, p, 1 << 28, 16, p, None) == 3


def test_decode_block_rejects_a_final_state_output(lib):
    dm = td.make_dims(B=1, S=16, d=256, Hq=4, Hkv=1, D=64, V=1024, Lmax=64, n_layers=0)
    p = ctypes.c_void_p(256)
    opts = td.td_step_opts(0, 0.0, td.td_paging(), 256)
    steps = ctypes.c_int(0)
    assert lib.td_decode_block(ctypes.byref(dm), None, None, p, p, p, p, 1, 16, 0.8,
                               ctypes.byref(opts), p, p, p, p, p, p, ctypes.byref(steps), p,
                               1 << 30, None) == 1
    # a misaligned final-state buffer is rejected by the step too
    opts.h_out = 258
    assert lib.td_denoise_step(ctypes.byref(dm), None, None, None, p, p, p, p, 1, 16, 0.8,
                               ctypes.byref(opts), p, p, p, p, p, p, p, 1 << 30, None) == 1


def test_unknown_attention_precision_is_rejected(lib):
    dm = td.make_dims(B=1, S=16, d=256, Hq=4, Hkv=1, D=64, V=1024, Lmax=64, n_layers=1)
    fake = ctypes.c_void_p(1 << 40)   # never dereferenced: the precision check fails first
    for bad in (2, -1):
        assert lib.td_block_attention(ctypes.byref(dm), fake, fake, fake, fake, fake, None, None,
                                      bad, fake, None, fake, 1 << 30, None) == 1


def test_decode_graph_form_is_a_host_setting(lib):
    # no graph has been built in this process: the form reads 0; unknown forms change nothing
    assert lib.td_decode_graph_form(0) == 0
    assert lib.td_decode_graph_form(7) == 0
    assert lib.td_decode_graph_form(1) == 0
