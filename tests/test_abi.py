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


_SCALER_OK = dict(num_blocks=2, num_workers=3, counts=0x10000, scale=0x20000, streak=0x30000,
                  backoff=0.5, growth=2.0, interval=4)


@pytest.mark.parametrize("kw,msg", [
    (dict(num_blocks=0), "num_blocks"),
    (dict(num_workers=0), "num_workers"),
    (dict(counts=0), "device pointers"),
    (dict(streak=0), "device pointers"),
    (dict(counts=0x10004), "aligned"),
    (dict(scale=0x20002), "aligned"),
    (dict(backoff=1.0), "backoff"),
    (dict(backoff=0.0), "backoff"),
    (dict(backoff=1e-50), "backoff"),
    (dict(growth=1e300), "growth"),
    (dict(growth=1.0), "growth"),
    (dict(growth=float("inf")), "growth"),
    (dict(interval=0), "interval"),
])
def test_scale_update_rejects_bad_arguments_before_any_launch(psgd, kw, msg):
    """Every argument error of psgd_scale_update returns PSGD_EINVAL with a message before
    anything is enqueued (no GPU is needed to see it)."""
    a = dict(_SCALER_OK, **kw)
    with pytest.raises(psgd.PSGDError) as ex:
        psgd.psgd_scale_update(a["num_blocks"], a["num_workers"], a["counts"], a["scale"],
                               a["streak"], a["backoff"], a["growth"], a["interval"], 0)
    assert ex.value.status == psgd.PSGD_EINVAL
    assert msg in str(ex.value), str(ex.value)


def test_clip_adam_workspace_and_argument_checks(psgd):
    """Sizes and argument errors of psgd_clip_adam, all answered before any launch."""
    ws = psgd.psgd_clip_adam_workspace_size([8192, 1, 0, 20000])
    assert ws > 0 and ws % 256 == 0
    assert ws >= 256 + 8 * (1 + 1 + 0 + 3)
    assert psgd.psgd_clip_adam_workspace_size([-1]) == 0
    assert psgd.psgd_clip_adam_workspace_size([1] * (psgd.PSGD_ADAM_MAX_TENSORS + 1)) == 0
    ok = dict(grads=[0x1000], params=[0x2000], exp_avg=[0x3000], exp_avg_sq=[0x4000],
              numel=[16], workspace_ptr=0x10000, ws_bytes=1 << 20, stream=0, lr=1e-3)
    for kw, msg in [(dict(lr=-1.0), "out of range"), (dict(beta1=1.0), "out of range"),
                    (dict(step=0), "out of range"), (dict(workspace_ptr=0x10010), "256-byte"),
                    (dict(ws_bytes=64), "workspace smaller"), (dict(params=[0x2002]), "aligned"),
                    (dict(skip_ptr=0x5000), "skip needs"),
                    (dict(skip_ptr=0x5000, block=[3], num_blocks=2), "block index")]:
        with pytest.raises(psgd.PSGDError) as ex:
            psgd.psgd_clip_adam(**dict(ok, **kw))
        assert ex.value.status == psgd.PSGD_EINVAL
        assert msg in str(ex.value), (kw, str(ex.value))


def test_reduce_uncompressed_argument_checks(psgd):
    """Argument errors of psgd_reduce_uncompressed, all answered before any launch."""
    ok = dict(in_ptrs=[0x1000, 0x2000], length=16, scale=1.0, out_ptr=0x3000, counts_ptr=0x4000)
    for kw, msg in [(dict(in_ptrs=[]), "num_workers"),
                    (dict(in_ptrs=[0x1000] * (psgd.PSGD_UNC_MAX_WORKERS + 1)), "num_workers"),
                    (dict(length=-1), "len"), (dict(scale=0.0), "scale"),
                    (dict(scale=float("inf")), "scale"), (dict(out_ptr=0x3004), "aligned"),
                    (dict(counts_ptr=0x4004), "aligned"), (dict(in_ptrs=[0x1000, 0x2008]), "aligned"),
                    (dict(in_ptrs=[0x1000, 0]), "NULL"), (dict(out_ptr=0), "required")]:
        with pytest.raises(psgd.PSGDError) as ex:
            psgd.psgd_reduce_uncompressed(**dict(ok, **kw))
        assert ex.value.status == psgd.PSGD_EINVAL
        assert msg in str(ex.value), (kw, str(ex.value))


def test_exchange_flag_planning_and_null_handles(psgd):
    """The data-parallel exchange calls: planning, rejections and NULL handles."""
    shapes = [(256, 512), (128, 64)]
    B, r = 3, 8
    plain, _ = psgd.make_config(shapes, B, 2, r, "f16")
    ex, _ = psgd.make_config(shapes, B, 2, r, "f16", flags=psgd.PSGD_FLAG_EXCHANGE)
    extra = psgd.psgd_workspace_size(ex) - psgd.psgd_workspace_size(plain)
    assert extra >= 4 * B * r * sum(m + n for m, n in shapes) + 8 * B
    bad, _ = psgd.make_config(shapes, B, 2, r, "f16", unc_len=16, flags=psgd.PSGD_FLAG_EXCHANGE)
    assert psgd.psgd_workspace_size(bad) == 0
    assert "unc_len == 0" in psgd.lib.psgd_last_error().decode()
    bad, _ = psgd.make_config(shapes, B, 2, r, "f16",
                              flags=psgd.PSGD_FLAG_EXCHANGE | psgd.PSGD_FLAG_STOP_AFTER_INGEST)
    assert psgd.psgd_workspace_size(bad) == 0
    lib = psgd.lib
    assert lib.psgd_step_p(None, None, None) == psgd.PSGD_EINVAL
    assert lib.psgd_step_q(None, None, None, 4, None) == psgd.PSGD_EINVAL
    assert lib.psgd_step_e(None, None, 4, None) == psgd.PSGD_EINVAL
    assert psgd.psgd_exchange_p(0, 0, 0) == 0 and psgd.psgd_exchange_q(0, 0, 0) == 0
    assert psgd.psgd_exchange_counts(0) == 0
