"""The native draft-depth gate (include/dmtp_gate.h, host code in libdmtp.so) against the
oracle (oracle/gate.py): the same seeded sequences of forwards, draft costs, settled
verifies and picks (both forms) give the same depths and values and the same state;
invalid arguments are refused with the gate unchanged. No GPU."""
import numpy as np
import pytest

from mtp_block_draft_gb300 import DmtpError, DmtpGate
from oracle.gate import DepthGate


def _same_state(native, ref):
    st = native.read()
    assert st["a"] == ref.a
    assert st["t"] == ref.T
    assert st["d"] == ref.d
    assert st["rho"] == ref.rho()
    assert st["picks"] == ref.picks and st["since_plain"] == ref.since_plain
    assert st["bin_judged"] == ref.bin_judged and st["bin_accepted"] == ref.bin_accepted


def _drive(seed, K, steps, priors=None):
    rng = np.random.default_rng(seed)
    native, ref = DmtpGate(K, priors), DepthGate(K, priors)
    picks = 0
    last_k = 0
    for _ in range(steps):
        op = rng.choice(["forward", "verify", "cost", "pick", "pick_p"],
                        p=[0.3, 0.25, 0.05, 0.25, 0.15])
        if op == "forward":
            rows = int(rng.integers(1, K + 2)) if rng.random() < 0.8 else 1
            sec = float(rng.uniform(0.5, 3.0)) * (1 + 0.1 * (rows - 1))
            native.forward(rows, sec)
            ref.forward(rows, sec)
        elif op == "cost":
            sec = float(rng.uniform(0.0, 0.4))
            native.draft_cost(sec)
            ref.draft_cost(sec)
        elif op == "verify":
            k = last_k if last_k > 0 else int(rng.integers(1, K + 1))
            accepted = int(rng.integers(0, k + 1))
            judged = accepted if accepted == k else accepted + 1
            p = rng.uniform(0, 1, judged).tolist() if rng.random() < 0.6 else None
            native.result(judged, accepted, p)
            ref.result(judged, accepted, p)
        elif op == "pick":
            proposed = int(rng.integers(0, K + 3))
            got, want = native.pick(proposed), ref.pick(proposed)
            assert got[0] == want[0]
            assert got[1] == want[1]
            last_k = got[0]
            picks += 1
        else:
            n = int(rng.integers(0, K + 1))
            p = rng.uniform(0, 1, n)
            p[rng.random(n) < 0.2] = rng.choice([0.0, 1.0, 0.1, 0.9])
            got, want = native.pick_p(p.tolist()), ref.pick_p(p.tolist())
            assert got[0] == want[0]
            assert got[1] == want[1]
            last_k = got[0]
            picks += 1
    _same_state(native, ref)
    native.close()
    return picks


@pytest.mark.parametrize("seed", range(12))
def test_native_gate_matches_oracle(seed):
    K = [7, 1, 3, 7, 12, 32][seed % 6]
    assert _drive(seed, K, 600) > 100


def test_native_gate_matches_oracle_with_priors():
    _drive(99, 7, 800, priors=[0.95, 0.9, 0.85, 0.8, 0.7, 0.6, 0.5])
    _drive(100, 4, 800, priors=[0.0, 0.0, 0.0, 0.0])


def test_long_run_forces_plain_steps_and_probes():
    """Only multi-row forwards: the plain step comes after 64 of them; probes every 16
    picks; both sides agree throughout."""
    native, ref = DmtpGate(7), DepthGate(7)
    for g in (native, ref):
        g.forward(1, 1.0)
    ks = []
    for i in range(300):
        a, b = native.pick(7), ref.pick(7)
        assert a == b
        ks.append(a[0])
        rows = a[0] + 1
        for g in (native, ref):
            g.forward(rows, 1.0 + 0.05 * (rows - 1))
        judged = min(a[0], 3)
        if a[0]:
            for g in (native, ref):
                g.result(judged, min(a[0], 2) if judged > 2 else judged)
    assert 0 in ks and max(ks) >= 1
    _same_state(native, ref)


def test_invalid_arguments_leave_the_gate_unchanged():
    native, ref = DmtpGate(5), DepthGate(5)
    for g in (native, ref):
        g.forward(1, 1.0)
        g.forward(3, 1.2)
        g.result(2, 1, [0.3, 0.8])
    before = native.read()
    bad = [lambda: native.forward(0, 1.0), lambda: native.forward(65, 1.0),
           lambda: native.forward(2, 0.0), lambda: native.forward(2, float("nan")),
           lambda: native.draft_cost(-1.0), lambda: native.draft_cost(float("inf")),
           lambda: native.result(3, 1), lambda: native.result(6, 5),
           lambda: native.result(2, 3), lambda: native.result(2, 1, [0.5, 1.5]),
           lambda: native.result(1, 0, [float("nan")]), lambda: native.pick(-1),
           lambda: native.pick_p([0.5, -0.1])]
    for f in bad:
        with pytest.raises(DmtpError):
            f()
    assert native.read() == before
    for bad_k, bad_p in ((0, None), (33, None), (3, [0.5, 2.0, 0.5])):
        with pytest.raises(DmtpError):
            DmtpGate(bad_k, bad_p)
    assert native.pick(5) == ref.pick(5)
