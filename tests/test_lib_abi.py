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
    inc = os.path.join(ROOT, "include")
    src = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc))
                  if f.endswith(".h"))
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


def _aligned_host_buffer(nbytes):
    """A 256-byte aligned host address; dmtp_init's failure paths below return before
    they touch the workspace or the device."""
    raw = ctypes.create_string_buffer(nbytes + 256)
    addr = (ctypes.addressof(raw) + 255) & ~255
    return raw, addr


def _init(lib, cfg, max_ctx, lens, ws_bytes, ws_addr=None):
    c = make_config(cfg, max_ctx)
    w = binding.dmtp_weights()
    n = len(lens)
    ids = (ctypes.c_int32 * max(1, sum(lens)))()
    plen = (ctypes.c_int32 * n)(*lens)
    raw = None
    if ws_addr is None:
        raw, ws_addr = _aligned_host_buffer(256)
    ctx = ctypes.c_void_p()
    r = lib.dmtp_init(ctypes.byref(c), ctypes.byref(w), ws_addr, ws_bytes, ids, plen, n,
                      None, ctypes.byref(ctx))
    del raw
    return r, ctx


def _ws_size(lib, cfg, max_ctx, batch):
    c = make_config(cfg, max_ctx)
    n = ctypes.c_size_t()
    assert lib.dmtp_workspace_size(ctypes.byref(c), batch, ctypes.byref(n)) == 0
    return n.value


def test_init_workspace_too_small_is_enomem(lib):
    """A workspace one byte short of dmtp_workspace_size: DMTP_ENOMEM, no context."""
    cfg = CONFIGS["b32"].replace(batch=3)
    need = _ws_size(lib, cfg, 1024, 3)
    r, ctx = _init(lib, cfg, 1024, [100, 37, 900], need - 1)
    assert r == -2 and not ctx.value


def test_init_prompt_past_capacity_is_ecapacity(lib):
    """A prompt that leaves no room for a round below max_ctx: DMTP_ECAPACITY before any
    launch, whatever the workspace."""
    cfg = CONFIGS["b32"].replace(batch=2)
    need = _ws_size(lib, cfg, 1024, 2)
    r, ctx = _init(lib, cfg, 1024, [100, 1024], need)
    assert r == -3 and not ctx.value


def test_init_rejects_empty_prompt_and_unaligned_workspace(lib):
    cfg = CONFIGS["b32"].replace(batch=2)
    need = _ws_size(lib, cfg, 1024, 2)
    r, ctx = _init(lib, cfg, 1024, [100, 0], need)
    assert r == -1 and not ctx.value
    raw, addr = _aligned_host_buffer(256)
    r, ctx = _init(lib, cfg, 1024, [100, 50], need, ws_addr=addr + 16)
    assert r == -1 and not ctx.value


def test_deterministic_option_and_error_word(lib):
    """deterministic takes 0 or 1 and adds the fixed-order K-part scratch to a bf16
    workspace; the error word of no context is 0."""
    cfg = CONFIGS["b32"]
    n0, n1 = ctypes.c_size_t(), ctypes.c_size_t()
    c = make_config(cfg, 5000)
    assert lib.dmtp_workspace_size(ctypes.byref(c), 32, ctypes.byref(n0)) == 0
    c.deterministic = 1
    assert lib.dmtp_workspace_size(ctypes.byref(c), 32, ctypes.byref(n1)) == 0
    assert n1.value > n0.value
    c.deterministic = 2
    assert lib.dmtp_workspace_size(ctypes.byref(c), 32, ctypes.byref(n1)) == -1
    lib.dmtp_error_word.restype = ctypes.c_uint32
    assert lib.dmtp_error_word(None) == 0


def test_workspace_size_grows_with_batch_and_context(lib):
    """Odd and even batches alike: more sequences or a longer context never need less."""
    cfg = CONFIGS["b32"]
    sizes = [_ws_size(lib, cfg.replace(batch=b), 2048, b) for b in (1, 2, 3, 5, 8)]
    assert all(a < b for a, b in zip(sizes, sizes[1:]))
    assert _ws_size(lib, cfg, 4096, 3) > _ws_size(lib, cfg, 2048, 3)


_C_GATE = r"""
#include <stdio.h>
#include "dmtp_gate.h"
int main(void) {
  dmtp_gate* g = NULL;
  if (dmtp_gate_create(7, NULL, &g) != DMTP_OK) return 1;
  const double p[7] = {0.93, 0.88, 0.4, 0.97, 0.12, 0.5, 0.99};
  for (int r = 0; r < 40; ++r) {
    int k = 0;
    double v = 0.0;
    if (dmtp_gate_forward(g, 1 + r % 8, 1.0 + 0.07 * (r % 8) + 0.001 * r) != DMTP_OK) return 2;
    if (r % 5 == 4 && dmtp_gate_draft_cost(g, 0.01 * r) != DMTP_OK) return 3;
    if (dmtp_gate_pick(g, 7, &k, &v) != DMTP_OK) return 4;
    printf("pick %d %.17g\n", k, v);
    if (dmtp_gate_pick_p(g, 7, p, &k, &v) != DMTP_OK) return 5;
    printf("pick_p %d %.17g\n", k, v);
    const int acc = r % 4, judged = acc + 1;
    if (dmtp_gate_result(g, judged, acc, p) != DMTP_OK) return 6;
  }
  dmtp_gate_stats st;
  if (dmtp_gate_read(g, &st) != DMTP_OK) return 7;
  printf("rho %.17g\n", st.rho);
  if (dmtp_gate_result(g, 3, 1, NULL) != DMTP_EINVAL) return 8;
  dmtp_gate_free(g);
  dmtp_gate_free(NULL);
  return 0;
}
"""


def test_headers_compile_as_c99_and_a_c_caller_runs_the_gate(lib, tmp_path):
    """include/*.h compile as strict C99; a C program linked against libdmtp.so drives
    the host-only gate and prints what the oracle computes for the same calls."""
    import shutil
    import subprocess
    from oracle.gate import DepthGate
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    inc = os.path.join(ROOT, "include")
    for h in sorted(os.listdir(inc)):
        src = tmp_path / f"hdr_{h}.c"
        src.write_text(f'#include "{h}"\nint main(void) {{ return 0; }}\n')
        subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", inc,
                        "-c", str(src), "-o", str(tmp_path / f"hdr_{h}.o")], check=True)
    src = tmp_path / "gate_caller.c"
    src.write_text(_C_GATE)
    libdir = os.path.dirname(binding.LIB_PATH)
    exe = tmp_path / "gate_caller"
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", inc, str(src), "-o", str(exe),
                    "-L", libdir, "-ldmtp", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.returncode
    got = out.stdout.split("\n")
    g = DepthGate(7)
    p = [0.93, 0.88, 0.4, 0.97, 0.12, 0.5, 0.99]
    want = []
    for r in range(40):
        g.forward(1 + r % 8, 1.0 + 0.07 * (r % 8) + 0.001 * r)
        if r % 5 == 4:
            g.draft_cost(0.01 * r)
        k, v = g.pick(7)
        want.append(f"pick {k} {v!r}")
        k, v = g.pick_p(p)
        want.append(f"pick_p {k} {v!r}")
        g.result(r % 4 + 1, r % 4, p)
    want.append(f"rho {g.rho()!r}")
    parsed = []
    for line in got[:len(want)]:
        name, *rest = line.split()
        vals = [rest[0], repr(float(rest[1]))] if name != "rho" else [repr(float(rest[0]))]
        parsed.append(" ".join([name] + vals))
    assert parsed == want
