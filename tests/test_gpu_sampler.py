"""Temperature / top-p sampling (qw_sample) against the oracle's sampler (needs a GB300).

The random numbers of the draw are inputs (seeded uniforms in (0, 1)), so the
kernel and the oracle draw with the same ones.  The token is an integer
decided by floating point: the kernel computes the Gumbel scores and the
nucleus masses in fp32, the oracle in float64.  So the test asks for the
oracle's token exactly, except on a row where a different token is equally
correct at fp32 precision: its score within 1e-4 of the best score (a
near-tie), or the nucleus boundary within 1e-5 of the mass target (a value
that one precision keeps and the other drops).  Those rows must hold a
valid token (one the looser of the two nuclei admits, scoring within the
tie margin of the best there), and at least 99 % of the rows must match
exactly.  Greedy rows (T = 0) must equal qw_argmax bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle as O
import seeded_inputs as si

pytestmark = pytest.mark.gpu

Z_TIE = 1e-4        # score margin below which two tokens are a near-tie at fp32 precision
MASS_TOL = 1e-5     # relative margin of the nucleus mass target


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_transformer_forward_gb300 import build
    build.build()
    from qwen3_transformer_forward_gb300 import _lib
    _lib.load()
    return _lib


def _valid_alternative(lg, T, P, u, tok):
    """True when tok is an fp32-precision-equivalent draw for this row (see module doc)."""
    z = lg / T
    e = np.exp(z - z.max())
    values = np.unique(lg)[::-1]
    mass = np.array([e[lg == c].sum() for c in values])
    cum = np.cumsum(mass)
    target = min(max(P, 0.0), 1.0) * cum[-1] if P > 0 else cum[-1]
    k_loose = int(np.argmax(cum >= target * (1 - MASS_TOL)))
    k_tight = int(np.argmax(cum >= min(target * (1 + MASS_TOL), cum[-1])))
    loose = lg >= values[max(k_loose, k_tight)]
    if not loose[tok]:
        return False
    score = np.where(loose, z - np.log(-np.log(u)), -np.inf)
    return score[tok] >= score.max() - Z_TIE * max(1.0, abs(score.max()))


def _ws_clean(ws, B):
    """Counters, histogram and row maxima (the parts a call must find zero) are zero."""
    return int(ws[:64 * 1024 + B * 65536 * 4 + B * 4].view(torch.int32).abs().sum()) == 0


def _run(L, logits, T, P, u):
    B, V = logits.shape
    out = torch.full((B,), -1, dtype=torch.int64, device="cuda")
    ws = torch.zeros(L.sample_workspace_size(B, V), dtype=torch.uint8, device="cuda")
    L.sample(logits.cuda(), torch.tensor(T, dtype=torch.float32, device="cuda"),
             torch.tensor(P, dtype=torch.float32, device="cuda"), u.cuda(), out, ws)
    torch.cuda.synchronize()
    L.device_error()
    return out.cpu().numpy(), ws


def _compare(logits, T, P, u, got, what):
    lg = logits.double().numpy()
    un = u.double().numpy()
    want = O.sample(lg, T, P, un)
    same = got == want
    for b in np.nonzero(~same)[0]:
        assert T[b] > 0, (what, b, "greedy rows must match exactly")
        assert _valid_alternative(lg[b], T[b], P[b], un[b], int(got[b])), (what, b, got[b], want[b])
    assert np.mean(same) >= 0.99, (what, float(np.mean(same)))
    return same


def test_sample_full_vocab_rows(L):
    """Eight rows of 151936 logits (the lm_head's shape), each with its own
    temperature and nucleus mass, greedy included."""
    B, V = 8, 151936
    logits = si.normal(0, "sample.full.logits", (B, V), 0.7, "bf16")
    u = si.uniform01(0, "sample.full.u", (B, V))
    T = [0.0, 0.5, 1.0, 1.0, 2.0, 0.8, 1e-3, 1.0]
    P = [1.0, 0.9, 0.95, 1.0, 0.5, 0.01, 1.0, 1e-6]
    got, ws = _run(L, logits, T, P, u)
    _compare(logits, T, P, u, got, "full vocab")
    # greedy row: the same token as qw_argmax
    ref = torch.empty(B, dtype=torch.int64, device="cuda")
    L.argmax(logits.cuda(), ref)
    torch.cuda.synchronize()
    assert int(ref[0]) == int(got[0])
    assert _ws_clean(ws, B)


def test_sample_many_rows_match_the_oracle_draws(L):
    """512 rows of 4096 logits with temperatures and nucleus masses spread over
    their ranges: the kernel's draws are the oracle's draws (a distribution
    check by construction: the oracle's frequencies are pinned on the CPU)."""
    B, V = 512, 4096
    logits = si.normal(0, "sample.many.logits", (B, V), 1.5, "bf16")
    u = si.uniform01(0, "sample.many.u", (B, V))
    T = (0.05 + 2.0 * si.uniform01(0, "sample.many.T", (B,))).tolist()
    P = si.uniform01(0, "sample.many.P", (B,)).tolist()
    T[::17] = [0.0] * len(T[::17])
    P[::13] = [1.0] * len(P[::13])
    got, _ = _run(L, logits, T, P, u)
    _compare(logits, T, P, u, got, "many rows")


def test_sample_ties_at_the_nucleus_boundary(L):
    """Logits from a few repeated values: the boundary value's tied tokens are all
    in the nucleus, whichever of them the draw picks."""
    B, V = 64, 2048
    levels = torch.tensor([3.0, 1.0, 1.0, 1.0, 0.0, -2.0], dtype=torch.bfloat16)
    pick = si.uniform_int(0, "sample.ties.pick", (B, V), 0, len(levels))
    logits = levels[pick]
    u = si.uniform01(0, "sample.ties.u", (B, V))
    T = [1.0] * B
    P = [0.2 + 0.6 * (b / B) for b in range(B)]
    got, _ = _run(L, logits, T, P, u)
    same = _compare(logits, T, P, u, got, "ties")
    assert same.all()


def test_sample_back_to_back_calls_reuse_the_workspace(L):
    """Two calls with different logits on one workspace: the second is not
    affected by the first's histogram or counters."""
    B, V = 16, 8192
    ws = torch.zeros(L.sample_workspace_size(B, V), dtype=torch.uint8, device="cuda")
    T = torch.full((B,), 0.9, device="cuda")
    P = torch.full((B,), 0.8, device="cuda")
    for name in ("sample.reuse.a", "sample.reuse.b"):
        logits = si.normal(0, name + ".logits", (B, V), 1.0, "bf16")
        u = si.uniform01(0, name + ".u", (B, V))
        out = torch.full((B,), -1, dtype=torch.int64, device="cuda")
        L.sample(logits.cuda(), T, P, u.cuda(), out, ws)
        torch.cuda.synchronize()
        L.device_error()
        _compare(logits, [0.9] * B, [0.8] * B, u, out.cpu().numpy(), name)
        assert _ws_clean(ws, B)
