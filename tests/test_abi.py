"""The C ABI loads and exports every entry point include/gk.h declares; host-only layout
functions agree with the closed form. No GPU work is launched here."""
import ctypes as ct
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "gk.h")
LIB = os.path.join(ROOT, "gpt_decoder_gb300", "libgk.so")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gk_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        from gpt_decoder_gb300.build import build

        build()
    return ct.CDLL(LIB)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 25
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_the_header(lib):
    from gpt_decoder_gb300 import gk

    assert set(declared_functions()) == set(gk.EXPORTED)


def test_flat_layout_tiles_the_buffer(lib):
    from gpt_decoder_gb300 import gk

    for (V, T, C, H, L) in ((64, 64, 96, 4, 4), (50257, 1024, 768, 12, 12), (7, 4, 8, 2, 2)):
        cfg = gk.gk_gpt_cfg(V, T, C, H, L)
        n = gk.gk_gpt_numel(cfg)
        assert n == V * C + T * C + L * (12 * C * C + 13 * C) + 2 * C
        assert gk.gk_gpt_n_decay(cfg) == V * C + T * C + L * 12 * C * C
        sizes = {gk.GK_T_LN1_W: C, gk.GK_T_LN1_B: C, gk.GK_T_ATTN_W: 3 * C * C, gk.GK_T_ATTN_B: 3 * C,
                 gk.GK_T_ATTNPROJ_W: C * C, gk.GK_T_ATTNPROJ_B: C, gk.GK_T_LN2_W: C, gk.GK_T_LN2_B: C,
                 gk.GK_T_FC_W: 4 * C * C, gk.GK_T_FC_B: 4 * C, gk.GK_T_MLPPROJ_W: 4 * C * C,
                 gk.GK_T_MLPPROJ_B: C}
        spans = [(gk.gk_gpt_offset(cfg, gk.GK_T_WTE, 0), V * C), (gk.gk_gpt_offset(cfg, gk.GK_T_WPE, 0), T * C),
                 (gk.gk_gpt_offset(cfg, gk.GK_T_LNF_W, 0), C), (gk.gk_gpt_offset(cfg, gk.GK_T_LNF_B, 0), C)]
        for l in range(L):
            for which, size in sizes.items():
                o = gk.gk_gpt_offset(cfg, which, l)
                spans.append((o, size))
                # matrices come first: AdamW's decay boundary is one index
                is_matrix = which in (gk.GK_T_ATTN_W, gk.GK_T_ATTNPROJ_W, gk.GK_T_FC_W, gk.GK_T_MLPPROJ_W)
                assert (o < gk.gk_gpt_n_decay(cfg)) == is_matrix
        spans.sort()
        pos = 0
        for o, size in spans:
            assert o == pos
            pos += size
        assert pos == n
        assert gk.gk_gpt_offset(cfg, gk.GK_T_ATTN_W, L) == -1
        assert gk.gk_gpt_offset(cfg, 99, 0) == -1
