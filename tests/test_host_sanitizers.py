"""The host-only units of the library (the draft-depth gate and the draft heads' token
list) under AddressSanitizer, UndefinedBehaviorSanitizer and LeakSanitizer: a driver
built from their sources with the sanitizers calls every entry point with seeded random
arguments, valid and invalid, and must exit cleanly. No GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "mtp_block_draft_gb300", "csrc")

DRIVER = r"""
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <vector>
#include "dmtp_gate.h"
#include "dmtp_vocab.h"

static uint64_t s = 0x9E3779B97F4A7C15ull;
static uint64_t next() { s ^= s << 13; s ^= s >> 7; s ^= s << 17; return s; }
static int rnd(int n) { return (int)(next() % (uint64_t)n); }
static double unif() { return (double)(next() >> 11) * (1.0 / 9007199254740992.0); }

#define EXPECT(c) do { if (!(c)) { std::printf("failed: %s line %d\n", #c, __LINE__); return 1; } } while (0)

int main() {
  // ---- gate ----
  dmtp_gate* g = nullptr;
  EXPECT(dmtp_gate_create(0, nullptr, &g) == DMTP_EINVAL && !g);
  EXPECT(dmtp_gate_create(DMTP_GATE_MAX_DRAFTS + 1, nullptr, &g) == DMTP_EINVAL);
  double bad_prior[3] = {0.5, NAN, 0.5};
  EXPECT(dmtp_gate_create(3, bad_prior, &g) == DMTP_EINVAL);
  EXPECT(dmtp_gate_create(3, nullptr, nullptr) == DMTP_EINVAL);
  for (int K = 1; K <= DMTP_GATE_MAX_DRAFTS; K += 7) {
    std::vector<double> pri(K);
    for (double& x : pri) x = unif();
    EXPECT(dmtp_gate_create(K, pri.data(), &g) == DMTP_OK);
    std::vector<double> p(DMTP_GATE_MAX_DRAFTS + 8);
    for (int it = 0; it < 4000; ++it) {
      for (double& x : p) x = unif();
      int k = -1;
      double v = 0;
      switch (rnd(9)) {
        case 0: dmtp_gate_forward(g, 1 + rnd(DMTP_GATE_MAX_ROWS + 3) - 1, 0.1 + unif()); break;
        case 1: dmtp_gate_draft_cost(g, unif() - 0.2); break;
        case 2: { int acc = rnd(K + 2) - 1, jud = acc + rnd(3) - 1;
                  dmtp_gate_result(g, jud, acc, rnd(2) ? p.data() : nullptr); break; }
        case 3: EXPECT(dmtp_gate_pick(g, rnd(K + 4), &k, rnd(2) ? &v : nullptr) == DMTP_OK);
                EXPECT(k >= 0 && k <= K); break;
        case 4: EXPECT(dmtp_gate_pick_p(g, rnd(K + 4), p.data(), &k, &v) == DMTP_OK);
                EXPECT(k >= 0 && k <= K); break;
        case 5: EXPECT(dmtp_gate_pick(g, -1, &k, &v) == DMTP_EINVAL);
                EXPECT(dmtp_gate_pick(g, 3, nullptr, &v) == DMTP_EINVAL);
                EXPECT(dmtp_gate_pick_p(g, 2, nullptr, &k, &v) == DMTP_EINVAL); break;
        case 6: EXPECT(dmtp_gate_forward(g, 2, NAN) == DMTP_EINVAL);
                EXPECT(dmtp_gate_forward(g, 0, 1.0) == DMTP_EINVAL);
                EXPECT(dmtp_gate_draft_cost(g, INFINITY) == DMTP_EINVAL); break;
        case 7: { p[0] = 1.5; EXPECT(dmtp_gate_pick_p(g, 1, p.data(), &k, &v) == DMTP_EINVAL);
                  EXPECT(dmtp_gate_result(g, 1, 0, p.data()) == DMTP_EINVAL); break; }
        default: { dmtp_gate_stats st;
                   EXPECT(dmtp_gate_read(g, &st) == DMTP_OK && st.max_drafts == K);
                   EXPECT(std::isfinite(st.rho)); }
      }
    }
    dmtp_gate_free(g);
  }
  dmtp_gate_free(nullptr);

  // ---- token list ----
  dmtp_vocab_list* l = nullptr;
  EXPECT(dmtp_vocab_create(0, 10, &l) == DMTP_EINVAL && !l);
  EXPECT(dmtp_vocab_create(10, -1, &l) == DMTP_EINVAL);
  EXPECT(dmtp_vocab_create(10, 1, nullptr) == DMTP_EINVAL);
  const int sizes[3] = {1, 300, 0};
  for (int si = 0; si < 3; ++si) {
    const int V = 5000;
    EXPECT(dmtp_vocab_create(V, sizes[si], &l) == DMTP_OK);
    std::vector<int32_t> toks(3000), ids(V);
    std::vector<uint8_t> mask(V);
    std::vector<int64_t> counts(V);
    for (int it = 0; it < 600; ++it) {
      const int n = rnd(2) ? rnd(8) : rnd(3000);
      for (int i = 0; i < n; ++i) toks[i] = rnd(4) ? rnd(50) : rnd(V);
      int listed = -1;
      switch (rnd(6)) {
        case 0: EXPECT(dmtp_vocab_begin_request(l, n ? toks.data() : nullptr, n, rnd(2)) == DMTP_OK); break;
        case 1: EXPECT(dmtp_vocab_picked(l, toks.data(), n % 9) == DMTP_OK); break;
        case 2: toks[0] = rnd(2) ? V : -1;
                EXPECT(dmtp_vocab_picked(l, toks.data(), 1 + n % 5) == DMTP_EINVAL);
                EXPECT(dmtp_vocab_begin_request(l, nullptr, 3, 0) == DMTP_EINVAL);
                EXPECT(dmtp_vocab_picked(l, toks.data(), -1) == DMTP_EINVAL); break;
        case 3: EXPECT(dmtp_vocab_ids(l, rnd(2) ? ids.data() : nullptr, &listed) == DMTP_OK);
                EXPECT(listed >= 1 && listed <= V); break;
        case 4: EXPECT(dmtp_vocab_mask(l, mask.data()) == DMTP_OK);
                EXPECT(dmtp_vocab_counts(l, counts.data()) == DMTP_OK); break;
        default: { dmtp_vocab_stats st;
                   EXPECT(dmtp_vocab_stats_read(l, &st) == DMTP_OK && st.vocab == V);
                   EXPECT(st.counted >= 0 && st.counted < DMTP_VOCAB_HALVE_EVERY); }
      }
    }
    dmtp_vocab_free(l);
  }
  dmtp_vocab_free(nullptr);
  std::printf("clean\n");
  return 0;
}
"""


def test_host_units_under_sanitizers(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    src = tmp_path / "driver.cpp"
    src.write_text(DRIVER)
    exe = tmp_path / "driver"
    cmd = [cxx, "-std=c++17", "-g", "-O1", "-fsanitize=address,undefined",
           "-fno-sanitize-recover=all", "-fno-omit-frame-pointer",
           "-I", os.path.join(ROOT, "include"), str(src),
           os.path.join(CSRC, "gate.cpp"), os.path.join(CSRC, "vocab.cpp"), "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 and "sanitize" in r.stderr:
        pytest.skip("sanitizer runtime not available: " + r.stderr[-200:])
    assert r.returncode == 0, r.stderr[-3000:]
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=0",
               UBSAN_OPTIONS="print_stacktrace=1")
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300, env=env)
    assert out.returncode == 0, (out.stdout[-2000:], out.stderr[-4000:])
    assert out.stdout.strip().endswith("clean")
