"""The oracle's SSD form (Mamba-2's state-space dual layer) against routes other than its own loop.

"Mamba 论文精读" (youngju.dev) §4.1 states the duality this form rests on: the
recurrence h_t = A_t h_{t-1} + B_t x_t, y_t = C_t h_t equals a masked matrix
product Y = (T o M) X, T the causal (lower-triangular) mask and M a
semiseparable matrix. With one decay a_t = exp(dt_t A_h) per head and step,
M[l, s] = (C_l . B_s) * prod_{r=s+1..l} a_r * dt_s. Pins:

* the matrix form itself, written with numpy from cumulative sums of dt * A
  (a sum of exponents instead of a running product), T = np.tril;
* the selective-scan oracle (pinned on its own) run on expanded inputs (A
  repeated over the head's channels and states, delta and bias over its
  channels) gives the same outputs and final state;
* the chunked form (masked products inside each chunk, the state passed from
  chunk to chunk) at chunk sizes 1, 7, 16 and 64, the decomposition a chunked
  GPU kernel computes, and the same with D x taken as D on the diagonal of the
  masked matrix;
* a sequence split in two and continued from the first part's final state.

Planted mistakes in copies of the C code must each fail one of these.
"""
import numpy as np
import pytest

import oracle


def problem(seed, batch=2, nheads=3, P=4, N=5, L=37, softplus=True, D=True, bias=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((batch, nheads * P, L))
    delta = rng.standard_normal((batch, nheads, L)) * 0.5 if softplus else rng.uniform(0.01, 0.3, (batch, nheads, L))
    A = -rng.uniform(0.3, 3.0, nheads)
    B = rng.standard_normal((batch, N, L))
    C = rng.standard_normal((batch, N, L))
    return dict(x=x, delta=delta, A=A, B=B, C=C, D=rng.standard_normal(nheads) if D else None,
                delta_bias=np.log(np.expm1(rng.uniform(0.02, 0.2, nheads))) if bias else None, softplus=softplus)


def eff_dt(p):
    d = p["delta"] + (0.0 if p["delta_bias"] is None else p["delta_bias"][None, :, None])
    return np.logaddexp(0.0, d) if p["softplus"] else d


def run(orc, p, h0=None):
    return orc.ssd(p["x"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["delta_bias"], p["softplus"], h0=h0)


def check_matrix_form(orc):
    p = problem(101)
    rng = np.random.default_rng(101)
    batch, dim, L = p["x"].shape
    H = p["A"].shape[0]
    P = dim // H
    h0 = rng.standard_normal((batch, H, P, p["B"].shape[1])) * 0.3
    y, hl = run(orc, p, h0)
    dt = eff_dt(p)
    for b in range(batch):
        for h in range(H):
            cum = np.cumsum(dt[b, h] * p["A"][h])                       # sum of dt*A up to l
            decay = np.exp(cum[:, None] - cum[None, :])                  # prod of a over (s, l]
            M = (p["C"][b].T @ p["B"][b]) * decay * dt[b, h][None, :]
            X = p["x"][b, h * P:(h + 1) * P].T                           # (L, P)
            want = np.tril(M) @ X + np.exp(cum)[:, None] * (p["C"][b].T @ h0[b, h].T)
            if p["D"] is not None:
                want = want + p["D"][h] * X
            np.testing.assert_allclose(y[b, h * P:(h + 1) * P].T, want, rtol=1e-11, atol=1e-11)
            Hend = (np.exp(cum[-1]) * h0[b, h]
                    + (X * (np.exp(cum[-1] - cum) * dt[b, h])[:, None]).T @ p["B"][b].T)
            np.testing.assert_allclose(hl[b, h], Hend, rtol=1e-11, atol=1e-11)


def check_scan_equivalence(orc):
    p = problem(102, softplus=True)
    batch, dim, L = p["x"].shape
    H = p["A"].shape[0]
    P = dim // H
    N = p["B"].shape[1]
    y, hl = run(orc, p)
    ys, hs = orc.scan(p["x"], np.repeat(p["delta"], P, axis=1), np.repeat(p["A"], P)[:, None].repeat(N, axis=1),
                      p["B"], p["C"], None if p["D"] is None else np.repeat(p["D"], P), None,
                      None if p["delta_bias"] is None else np.repeat(p["delta_bias"], P), p["softplus"])
    np.testing.assert_allclose(y.reshape(batch * dim, L), ys, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hl.reshape(batch * dim, N), hs, rtol=1e-12, atol=1e-13)


def chunked(p, Q, h0=None):
    """The chunked SSD form in fp64: masked products within chunks, states passed between them."""
    x, B, C, A = p["x"], p["B"], p["C"], p["A"]
    batch, dim, L = x.shape
    H = A.shape[0]
    P = dim // H
    N = B.shape[1]
    dt = eff_dt(p)
    y = np.zeros_like(x)
    hl = np.zeros((batch, H, P, N))
    for b in range(batch):
        for h in range(H):
            S = np.zeros((P, N)) if h0 is None else h0[b, h].copy()
            for l0 in range(0, L, Q):
                sl = slice(l0, min(L, l0 + Q))
                d = dt[b, h, sl]
                cum = np.cumsum(d * A[h])
                X = x[b, h * P:(h + 1) * P, sl].T
                Cc, Bc = C[b][:, sl], B[b][:, sl]
                G = np.tril((Cc.T @ Bc) * np.exp(cum[:, None] - cum[None, :]) * d[None, :])
                Y = G @ X + np.exp(cum)[:, None] * (Cc.T @ S.T)
                if p["D"] is not None:
                    Y = Y + p["D"][h] * X
                y[b, h * P:(h + 1) * P, sl] = Y.T
                S = np.exp(cum[-1]) * S + (X * (np.exp(cum[-1] - cum) * d)[:, None]).T @ Bc.T
            hl[b, h] = S
    return y, hl


def check_chunked_form(orc):
    p = problem(103, L=70, softplus=False, bias=False)
    y, hl = run(orc, p)
    for Q in (1, 7, 16, 64):
        yc, hc = chunked(p, Q)
        np.testing.assert_allclose(yc, y, rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(hc, hl, rtol=1e-10, atol=1e-11)


def check_skip_in_the_diagonal(orc):
    # the skip term D x_l as D on the diagonal of the masked intra-chunk matrix
    # (the GPU kernel's form): Y = (T o M + D I) X over each chunk, nothing added after
    p = problem(105, L=70)
    y, hl = run(orc, p)
    x, B, C, A = p["x"], p["B"], p["C"], p["A"]
    batch, dim, L = x.shape
    H = A.shape[0]
    P = dim // H
    dt = eff_dt(p)
    for b in range(batch):
        for h in range(H):
            S = np.zeros((P, B.shape[1]))
            for l0 in range(0, L, 32):
                sl = slice(l0, min(L, l0 + 32))
                d = dt[b, h, sl]
                cum = np.cumsum(d * A[h])
                X = x[b, h * P:(h + 1) * P, sl].T
                Cc, Bc = C[b][:, sl], B[b][:, sl]
                G = np.tril((Cc.T @ Bc) * np.exp(cum[:, None] - cum[None, :]) * d[None, :])
                G = G + p["D"][h] * np.eye(len(d))
                Y = G @ X + np.exp(cum)[:, None] * (Cc.T @ S.T)
                np.testing.assert_allclose(Y.T, y[b, h * P:(h + 1) * P, sl], rtol=1e-10, atol=1e-11)
                S = np.exp(cum[-1]) * S + (X * (np.exp(cum[-1] - cum) * d)[:, None]).T @ Bc.T
            np.testing.assert_allclose(S, hl[b, h], rtol=1e-10, atol=1e-11)


def check_split_continuation(orc):
    p = problem(104, L=41)
    y, hl = run(orc, p)
    for cut in (1, 16, 40):
        a = {k: (v[..., :cut] if isinstance(v, np.ndarray) and v.ndim == 3 else v) for k, v in p.items()}
        c = {k: (v[..., cut:] if isinstance(v, np.ndarray) and v.ndim == 3 else v) for k, v in p.items()}
        y1, h1 = run(orc, a)
        y2, h2 = run(orc, c, h1)
        np.testing.assert_allclose(np.concatenate([y1, y2], axis=2), y, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(h2, hl, rtol=1e-12, atol=1e-13)


CHECKS = [check_matrix_form, check_scan_equivalence, check_chunked_form, check_skip_in_the_diagonal,
          check_split_continuation]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check(oracle.default())


def test_rejects_zoh_flag():
    # the ZOH gain is a feature of the per-state scan; the SSD form refuses it
    rc = oracle.default().lib.oracle_ssd(1, 1, 1, 1, 0, None, None, None, None, None, None, None, None,
                                         oracle.ZOH, None, None)
    assert rc == -3


MUTANTS = {
    "channel = p * nheads + h (heads interleaved)": ("const int64_t i = (b * dim + h * headdim + p) * seqlen + l;",
                                                    "const int64_t i = (b * dim + p * nheads + h) * seqlen + l;"),
    "decay after the input term": ("*hp = a * (*hp) + dt * Bb[n * seqlen + l] * xv;",
                                   "*hp = a * ((*hp) + dt * Bb[n * seqlen + l] * xv);"),
    "dt missing from the input term": ("*hp = a * (*hp) + dt * Bb[n * seqlen + l] * xv;",
                                       "*hp = a * (*hp) + Bb[n * seqlen + l] * xv;"),
    "readout before the update": ("                        *hp = a * (*hp) + dt * Bb[n * seqlen + l] * xv;\n"
                                  "                        acc += Cb[n * seqlen + l] * (*hp);",
                                  "                        acc += Cb[n * seqlen + l] * (*hp);\n"
                                  "                        *hp = a * (*hp) + dt * Bb[n * seqlen + l] * xv;"),
    "skip term of head 0 for every head": ("if (Dskip) acc += Dskip[h] * xv;", "if (Dskip) acc += Dskip[0] * xv;"),
    "bias of head 0 for every head": ("if (bias) dt += bias[h];", "if (bias) dt += bias[0];"),
    "state carried from head to head": ("for (int64_t i = 0; i < headdim * dstate; ++i) H[i] = h0 ? h0[s0 + i] : 0.0;",
                                        "if (h == 0) for (int64_t i = 0; i < headdim * dstate; ++i) H[i] = h0 ? h0[s0 + i] : 0.0;"),
    "B used as C in the readout": ("acc += Cb[n * seqlen + l] * (*hp);", "acc += Bb[n * seqlen + l] * (*hp);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(before) >= 1, f"mutation site for '{name}' not found"
    (tmp_path / "mutant.c").write_text(src.replace(before, after))
    orc = oracle.Oracle(oracle.build(str(tmp_path / "mutant.c"), str(tmp_path / "libmutant.so")))
    failed = []
    for check in CHECKS:
        try:
            check(orc)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"mutant '{name}' passes every pin"
