"""The C-ABI library builds for sm_103a, loads, exports every function that
include/dmtp.h declares, and rejects bad configurations on the host (no GPU)."""
import ctypes
import os
import re

import pytest

from mtp_block_draft_gb300 import binding, build, load_library, make_config
from synth import CONFIGS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "dmtp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dmtp_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert set(names) == set(binding.EXPORTS), names
    for n in names:
        assert getattr(lib, n) is not None


def test_strerror(lib):
    for code in range(0, -7, -1):
        assert lib.dmtp_strerror(code)
    assert b"unknown" in lib.dmtp_strerror(-99)


@pytest.mark.parametrize("name", list(CONFIGS))
def test_workspace_size_all_configs(lib, name):
    cfg = CONFIGS[name]
    c = make_config(cfg, cfg.ctx_hi + 8 * 40)
    n = ctypes.c_size_t()
    assert lib.dmtp_workspace_size(ctypes.byref(c), cfg.batch, ctypes.byref(n)) == 0
    assert n.value > 0


def test_rejects_bad_configs(lib):
    cfg = CONFIGS["b32"]
    n = ctypes.c_size_t()
    c = make_config(cfg, 5000)
    assert lib.dmtp_workspace_size(ctypes.byref(c), 33, ctypes.byref(n)) == -1   # B*8 > 256
    c = make_config(cfg, 5000)
    c.n_kv_heads = 3
    assert lib.dmtp_workspace_size(ctypes.byref(c), 32, ctypes.byref(n)) == -1   # hq % hkv
    c = make_config(cfg.replace(d_model=2040), 5000)
    assert lib.dmtp_workspace_size(ctypes.byref(c), 32, ctypes.byref(n)) == -1   # K % 64 (bf16)
    c = make_config(cfg, 5000)
    c.mask_id = cfg.vocab
    assert lib.dmtp_workspace_size(ctypes.byref(c), 32, ctypes.byref(n)) == -1
    assert lib.dmtp_workspace_size(None, 32, ctypes.byref(n)) == -1


def test_init_rejects_null_arguments(lib):
    ctx = ctypes.c_void_p()
    assert lib.dmtp_init(None, None, None, 0, None, None, 1, None, ctypes.byref(ctx)) == -1
    assert not ctx.value
    lib.dmtp_free(None)   # NULL is a no-op
