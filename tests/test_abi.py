"""The C-ABI library loads and exports every entry point psgd.h declares, and its host-
side validation and planning behave, all without a GPU (no compute calls here)."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "psgd.h")


@pytest.fixture(scope="module")
def psgd():
    from rank_gradient_compression_gb300 import build
    build.build()
    from rank_gradient_compression_gb300 import psgd as mod
    return mod


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(psgd_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports(psgd):
    assert declared_functions() == sorted(psgd.EXPORTS)


def test_library_exports_every_declared_symbol(psgd):
    out = subprocess.run(["nm", "-D", "--defined-only", psgd.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (psgd_\w+)", out))
    missing = [f for f in declared_functions() if f not in exported]
    assert not missing, missing
    for f in declared_functions():
        assert hasattr(psgd.lib, f)


def test_strerror(psgd):
    assert psgd.psgd_strerror(psgd.PSGD_OK) == "ok"
    assert "timed out" in psgd.psgd_strerror(psgd.PSGD_ETIMEOUT)


@pytest.mark.parametrize("kw,msg", [
    (dict(shapes=[(64, 30)], dtype="f16"), "multiple of 16"),
    (dict(shapes=[(64, 32)], dtype="f16", rank=40), "rank must be"),
    (dict(shapes=[(64, 32)], dtype="f16", rank=0), "rank must be"),
    (dict(shapes=[(0, 32)], dtype="f16"), "positive"),
    (dict(shapes=[(64, 32)], dtype="f16", workers=0), ">= 1"),
    (dict(shapes=[(64, 32)], dtype="f16", skip_fraction=0.0), "skip_fraction"),
    (dict(shapes=[(2048, 2048)], dtype="f16", rank=1100), "above 1024"),
])
def test_invalid_configs_are_rejected(psgd, kw, msg):
    args = dict(blocks=1, workers=2, rank=4, unc_len=0, skip_fraction=1.0)
    args.update(kw)
    cfg, _ = psgd.make_config(args.pop("shapes"), args["blocks"], args["workers"], args["rank"],
                              args.pop("dtype"), args["unc_len"], args["skip_fraction"])
    assert psgd.psgd_workspace_size(cfg) == 0
    assert msg in psgd.lib.psgd_last_error().decode()


def test_ranks_above_128_are_planned(psgd):
    """Ranks above the tensor engine's 128 (up to 1024) get a workspace: the FFMA engine
    runs them, with the orthonormalisation in 128-column blocks."""
    cfg, _ = psgd.make_config([(1024, 2048)], 1, 2, 896, "f16")
    assert psgd.psgd_workspace_size(cfg) > 0


def test_workspace_and_mask_layout(psgd):
    shapes = [(3968, 1488), (3968, 496), (3968, 1984), (15872, 496)]
    cfg, _ = psgd.make_config(shapes, 2, 8, 112, "f16")
    ws = psgd.psgd_workspace_size(cfg)
    # M scratch alone: W * sum(mn) * 2 bytes per block
    assert ws >= 2 * 8 * sum(m * n for m, n in shapes) * 2
    words = psgd.psgd_mask_words(cfg)
    assert words == 2 * 8 * sum((m * n + 31) // 32 for m, n in shapes)
    offs = sorted(psgd.psgd_mask_offset(cfg, b, j, w) for b in range(2) for j in range(4) for w in range(8))
    assert offs[0] == 0 and len(set(offs)) == len(offs) and offs[-1] < words
    assert psgd.psgd_mask_offset(cfg, 2, 0, 0) == -1


def test_no_cpu_fallback_when_library_missing(tmp_path):
    """The binding raises when the shared library is absent: no silent fallback."""
    code = ("import os; os.environ['PSGD_LIB'] = '/nonexistent/libpsgd.so'\n"
            "try:\n import rank_gradient_compression_gb300.psgd\nexcept ImportError as e:\n print('raised')\n")
    r = subprocess.run(["python", "-c", code], capture_output=True, text=True, cwd=ROOT)
    assert "raised" in r.stdout
