"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, and refuses bad arguments synchronously (no CUDA call is
reached for any case here)."""
import ctypes as C
import os
import re

import pytest

import moe_speculative_verify_gb300 as m
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_verify.h")


@pytest.fixture(scope="module")
def lib():
    m.build()
    return m.load()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:size_t|moe_status_t|const char\*)\s+(moe_\w+)\(",
                                 text, re.M)))


# The boundary's entry points as the hot-path scope lists them; the header
# declares each of them (plus the stepwise calls and the extensions).
SCOPE_ENTRY_POINTS = {"moe_route", "moe_build_union", "moe_expert_ffn_fp8", "moe_combine",
                      "moe_layer", "moe_workspace_size", "moe_get_device_error",
                      "moe_status_string"}


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert SCOPE_ENTRY_POINTS <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_size_query(lib):
    cfg = _cfg()
    for R in (0, 1, 8, 64, 65, 512, 4096):
        assert m.moe_workspace_size(cfg, R) == m.moe_workspace_bytes(cfg, R)
        # one buffer of that size also holds a union and an FFN workspace
        assert m.moe_workspace_size(cfg, R) >= m.moe_union_bytes(cfg, R)
        assert m.moe_workspace_size(cfg, R) >= m.moe_ffn_workspace_bytes(cfg, R)
    n = C.c_size_t(77)
    assert lib.moe_workspace_size(C.byref(cfg), m.MOE_MAX_ROWS + 1, C.byref(n)) == 2
    assert n.value == 0
    assert lib.moe_workspace_size(C.byref(cfg), -1, C.byref(n)) == 1
    assert lib.moe_workspace_size(C.byref(_cfg(hidden=100)), 8, C.byref(n)) == 1
    assert lib.moe_workspace_size(None, 8, C.byref(n)) == 1
    assert lib.moe_workspace_size(C.byref(cfg), 8, None) == 1


def test_noalloc_row_limit_at_glm_shape(lib):
    """The no-allocation entry point's fixed 32 MiB array holds the workspace of
    up to 109 rows at the GLM-5.2 shape, and not of 110 (the limit stated beside
    the entry point)."""
    cfg = _cfg()
    assert m.moe_workspace_bytes(cfg, 109) <= 32 << 20 < m.moe_workspace_bytes(cfg, 110)


def test_status_strings(lib):
    assert m.moe_status_string(0) == "MOE_OK"
    assert m.moe_status_string(4) == "MOE_ERR_TIMEOUT"
    assert m.moe_status_string(99) == "MOE_ERR_UNKNOWN"


def _cfg(**kw):
    c = m.Config.from_shape(synth.GLM52)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


FAKE = 1 << 40     # never dereferenced: every call below is refused or has R == 0


def _route(lib, cfg, R, x=FAKE, wr=FAKE, bias=FAKE, ids=FAKE, w=FAKE, logits=FAKE):
    return lib.moe_route(C.byref(cfg) if cfg is not None else None, x, wr, bias, None, R, ids, w,
                         logits, None)


def test_route_refusals(lib):
    assert _route(lib, None, 8) == 1
    assert _route(lib, _cfg(hidden=6000), 8) == 1              # not a multiple of 128
    assert _route(lib, _cfg(inter=100), 8) == 1
    assert _route(lib, _cfg(n_groups=7), 8) == 1               # 256 % 7 != 0
    assert _route(lib, _cfg(topk_groups=9), 8) == 1            # TG > G
    assert _route(lib, _cfg(topk=200), 8) == 1                 # K > TG * E / G
    assert _route(lib, _cfg(n_experts=512, n_groups=8), 8) == 2
    assert _route(lib, _cfg(hidden=32768), 8) == 2
    assert _route(lib, _cfg(n_shared=2), 8) == 2
    assert _route(lib, _cfg(), -1) == 1
    assert _route(lib, _cfg(), m.MOE_MAX_ROWS + 1) == 2       # no silent truncation
    assert _route(lib, _cfg(), 8, x=None) == 1
    assert _route(lib, _cfg(), 8, logits=None) == 1
    assert _route(lib, _cfg(), 8, x=FAKE + 2) == 1             # misaligned bf16 array
    assert _route(lib, _cfg(), 8, wr=FAKE + 4) == 1
    assert _route(lib, _cfg(), 0) == 0                         # R == 0: nothing launched


def test_union_and_layer_refusals(lib):
    cfg = _cfg()
    need = m.moe_union_bytes(cfg, 64)
    assert need > 0
    assert lib.moe_build_union(C.byref(cfg), FAKE, 64, FAKE, need - 4, None) == 5
    assert lib.moe_build_union(C.byref(cfg), FAKE, 64, FAKE + 4, need, None) == 1
    assert lib.moe_build_union(C.byref(cfg), FAKE, 0, FAKE, need, None) == 0
    wts = m.Weights(*([FAKE] * 12))
    wsb = m.moe_workspace_bytes(cfg, 8)
    assert wsb > 0
    args = [C.byref(cfg), FAKE, FAKE, FAKE, C.byref(wts), None, 8, FAKE, None, None, FAKE]
    assert lib.moe_layer(*args, wsb - 1, None) == 5
    assert lib.moe_layer(*args[:10], FAKE + 16, wsb, None) == 1      # workspace not 256-aligned
    bad = m.Weights(*([FAKE] * 12))
    bad.s_down = None                                                  # unscaled fp8 refused
    assert lib.moe_layer(C.byref(cfg), FAKE, FAKE, FAKE, C.byref(bad), None, 8, FAKE, None, None,
                         FAKE, wsb, None) == 1
    bad2 = m.Weights(*([FAKE] * 12))
    bad2.w_up = FAKE + 8                                               # TMA needs 16-byte alignment
    assert lib.moe_layer(C.byref(cfg), FAKE, FAKE, FAKE, C.byref(bad2), None, 8, FAKE, None, None,
                         FAKE, wsb, None) == 1
    assert lib.moe_layer(C.byref(cfg), FAKE, FAKE, FAKE, C.byref(wts), None, 0, FAKE, None, None,
                         FAKE, wsb, None) == 0
    ffn_b = m.moe_ffn_workspace_bytes(cfg, 8)
    assert lib.moe_expert_ffn_fp8(C.byref(cfg), FAKE, C.byref(wts), FAKE, 8, FAKE, FAKE, FAKE,
                                  ffn_b - 1, None) == 5
    assert lib.moe_combine(C.byref(cfg), FAKE, None, FAKE, FAKE, 8, FAKE, None) == 1  # S=1 needs y_shared
    assert lib.moe_diag_wait_timeout(FAKE, 0, None) == 1


def test_tile_weights_refusals(lib):
    f = lib.moe_tile_weights
    assert f(FAKE, FAKE + 4096, 2, 256, 256, None) == 1          # overlapping
    assert f(FAKE + 8, FAKE << 1, 1, 256, 256, None) == 1        # src not 16-byte aligned
    assert f(FAKE, (FAKE << 1) + 4, 1, 256, 256, None) == 1      # dst not 16-byte aligned
    assert f(FAKE, FAKE << 1, 1, 200, 256, None) == 1            # rows not a multiple of 128
    assert f(FAKE, FAKE << 1, 1, 256, 16384 + 128, None) == 1    # cols above 16384
    assert f(FAKE, FAKE << 1, -1, 256, 256, None) == 1
    assert f(None, FAKE << 1, 1, 256, 256, None) == 1
    assert f(FAKE, FAKE << 1, 0, 256, 256, None) == 0            # nothing to do
    cfg = _cfg()
    wsb = m.moe_workspace_bytes(cfg, 8)
    bad = m.Weights(*([FAKE] * 12), 2)                           # unknown layout
    assert lib.moe_layer(C.byref(cfg), FAKE, FAKE, FAKE, C.byref(bad), None, 8, FAKE, None, None,
                         FAKE, wsb, None) == 1


def test_ffn_layout_mirror_matches_library(lib):
    """The binding's mirror of the FFN workspace carve-up (which the GPU tests
    use to read regions of the workspace) ends where the library's size query
    says, for every tile width, with and without a shared expert."""
    import dataclasses
    for sh in (synth.GLM52, synth.TINY, dataclasses.replace(synth.TINY, n_shared=0)):
        cfg = m.Config.from_shape(sh)
        for R in (1, 8, 63, 64, 65, 512, 513, 4096):
            lay = m.ffn_layout(cfg, R)
            assert lay["bytes"] == m.moe_ffn_workspace_bytes(cfg, R), (sh, R)
            assert lay["ready"] < lay["sched"] < lay["xg"] < lay["xs"] < lay["hq"] < lay["hs"]


def test_sizes(lib):
    cfg = _cfg()
    for R in (1, 8, 64, 512, 4096):
        ub = m.moe_union_bytes(cfg, R)
        lay = m.union_layout(cfg, R)
        assert ub >= (lay["items"] + 4 * (R * 9 // 16 + min(256, R * 8) + 2)) * 4
        ffn = m.moe_ffn_workspace_bytes(cfg, R)
        # gathered activations and h: (R*(K+1)) rows of H and I bytes at least
        assert ffn >= R * 9 * (6144 + 2048)
        assert m.moe_workspace_bytes(cfg, R) >= ffn + ub + R * 8 * 6144 * 4
    assert m.moe_workspace_bytes(cfg, m.MOE_MAX_ROWS + 1) == 0
    assert m.moe_union_bytes(_cfg(hidden=100), 8) == 0
