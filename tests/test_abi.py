"""The C-ABI library builds, loads and exports every entry point its header
declares; host-side argument checks reject bad calls before anything reaches
the GPU (so these run without one)."""

import ctypes
import os
import re

import pytest

import paged_gqa_decode_reshape_gb300 as pg
import paged_gqa_decode_reshape_gb300.build as pgb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "paged_decode.h")


@pytest.fixture(scope="module")
def lib():
    pgb.build()
    return pg.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:PA_API\s+)?(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_pages_entry_points():
    names = declared_functions()
    for n in ["pa_reshape_and_cache", "pa_decode", "quest_update_meta", "quest_select_topk",
              "quest_sparse_decode"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in paged_decode.h but not exported"


def test_binding_wraps_every_entry_point():
    """Every C entry point has a same-named Python wrapper in the binding (argument
    marshalling only). pa_last_cuda_error feeds the binding's error messages, and
    pa_decode_no_alloc (with its status query) is for C callers that must not
    allocate."""
    for n in declared_functions():
        if n in ("pa_last_cuda_error", "pa_decode_no_alloc", "pa_decode_no_alloc_status"):
            continue
        assert n in pg.__all__ and callable(getattr(pg, n, None)), f"{n} has no Python wrapper"


def test_status_strings(lib):
    assert pg.pa_status_string(0) == "PA_OK"
    assert pg.pa_status_string(-1) == "PA_ERR_INVALID_ARG"
    assert pg.pa_status_string(-3) == "PA_ERR_WORKSPACE"
    assert pg.pa_status_string(12345) == "PA_ERR_UNKNOWN"


def _decode(lib, **over):
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: checks fail first
    args = dict(out=fake, q=fake, kc=fake, vc=fake, bt=fake, MBS=4, ctx=fake, B=2, Hq=28, Hkv=4,
                D=128, BS=16, NB=64, scale=0.088, ws=fake, ws_bytes=1 << 30, stream=None)
    args.update(over)
    return lib.pa_decode(args["out"], args["q"], args["kc"], args["vc"], args["bt"], args["MBS"],
                         args["ctx"], args["B"], args["Hq"], args["Hkv"], args["D"], args["BS"],
                         args["NB"], args["scale"], args["ws"], args["ws_bytes"], args["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(q=None), -1),
    (dict(out=None), -1),
    (dict(ws=None), -1),
    (dict(Hq=30), -1),                  # Hq not a multiple of Hkv
    (dict(B=0), -1),
    (dict(scale=-1.0), -1),
    (dict(D=96), -2),                   # unsupported head_dim
    (dict(BS=32), -2),                  # unsupported block size
    (dict(Hq=36, Hkv=4), -2),           # group of 9 query heads
    (dict(B=5000), -2),                 # batch above the supported maximum
    (dict(q=ctypes.c_void_p((1 << 20) + 2)), -1),   # misaligned pointer
])
def test_decode_rejects_bad_arguments_on_host(lib, over, status):
    assert _decode(lib, **over) == status


def test_reshape_zero_tokens_is_a_noop(lib):
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 0, 4, 128, 16, 10, None) == 0
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 5, 4, 128, 16, 10, None) == -1
    assert lib.quest_update_meta(None, None, None, None, 0, 4, 128, 16, 10, None) == 0


def test_select_workspace_size_and_checks(lib):
    assert pg.quest_select_workspace_size(16, 4, 1024) == 16 * 4 * 1024 * 4
    assert pg.quest_select_workspace_size(0, 4, 1024) == 0
    fake = ctypes.c_void_p(1 << 20)
    need = pg.quest_select_workspace_size(2, 4, 8)
    rc = lib.quest_select_topk(fake, fake, fake, fake, fake, 8, fake, 2, 28, 4, 128, 16, 64, 4,
                               fake, need - 1, None)
    assert rc == -3
    rc = lib.quest_select_topk(fake, fake, fake, fake, fake, 8, fake, 2, 28, 4, 128, 16, 64, 0,
                               fake, need, None)
    assert rc == -1


def test_dense_budget_rejects_a_negative_budget(lib):
    fake = ctypes.c_void_p(1 << 20)
    rc = lib.pa_decode_budget(fake, fake, fake, fake, fake, 4, fake, 2, 28, 4, 128, 16, 64, 0.088, -1,
                              fake, 1 << 30, None)
    assert rc == -1


def test_sparse_requires_selection(lib):
    fake = ctypes.c_void_p(1 << 20)
    rc = lib.quest_sparse_decode(fake, fake, fake, fake, fake, 4, fake, None, 4, 2, 28, 4, 128, 16,
                                 64, 0.088, fake, 1 << 30, None)
    assert rc == -1


def test_product_package_does_not_touch_the_oracle():
    """The product path never imports the CPU oracle."""
    pkg = os.path.join(ROOT, "paged_gqa_decode_reshape_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", src, flags=re.M), f
                assert "liboracle" not in src, f


def test_fp8_entry_points_check_arguments_on_host(lib):
    """The 8-bit cache entry points take head_dim 128 only and need both
    scale arrays; both are rejected before anything is launched."""
    fake = ctypes.c_void_p(1 << 20)
    dec = lambda D, ks: lib.pa_decode_fp8(fake, fake, fake, fake, ks, fake, fake, 4, fake, 2, 28, 4, D,
                                          16, 64, 0.088, fake, 1 << 30, None)
    assert dec(64, fake) == -2
    assert dec(128, None) == -1
    assert lib.quest_sparse_decode_fp8(fake, fake, fake, fake, fake, fake, fake, 4, fake, None, 4, 2,
                                       28, 4, 128, 16, 64, 0.088, fake, 1 << 30, None) == -1
    assert lib.pa_reshape_and_cache_fp8(fake, fake, fake, fake, fake, 3, fake, fake, 4, 64, 16, 10,
                                        None) == -2
    assert lib.pa_reshape_and_cache_fp8(fake, fake, fake, fake, fake, 3, None, fake, 4, 128, 16, 10,
                                        None) == -1
    assert lib.pa_reshape_and_cache_fp8(None, None, None, None, None, 0, None, None, 4, 128, 16, 10,
                                        None) == 0
    assert lib.quest_reshape_and_cache_fp8(fake, fake, fake, fake, None, fake, fake, 3, fake, fake, 4,
                                           128, 16, 10, None) == -1
    need = pg.quest_select_workspace_size(2, 4, 8)
    assert lib.quest_select_topk_fp8(fake, fake, fake, fake, fake, 8, fake, 2, 28, 4, 64, 16, 64, 4,
                                     fake, need, None) == -2
    assert lib.quest_select_topk_fp8(fake, fake, fake, fake, fake, 8, fake, 2, 28, 4, 128, 16, 64, 4,
                                     fake, need - 1, None) == -3
