"""The chunk form of the scan's backward, restated on the CPU in fp64, against
the per-step backward oracle (itself pinned by finite differences).

The backward kernels evaluate the gradients chunk by chunk as dense
contractions; this test writes those contractions out (no CUDA code is used)
and checks that they are the derivatives of the recurrence. Within a chunk
with inclusive cumsum cs of dt a, entering state h_in and G_out, the gradient
at the chunk's last state through the later steps only:

* chains: h_in(c+1) = e^{cs_last} h_in(c) + S(c), S(c) = sum_j e^{cs_last - cs_j} dt_j B_j x_j^T;
  G_out(c-1) = e^{cs_last} G_out(c) + R(c), R(c) = sum_s e^{cs_s} C_s dy_s^T; d init = G_out(-1);
* with CB = C B^T, DX = dy x^T, E = causal e^{cs_i - cs_j}, Mt = E o CB, A2 = E o DX:
  dx = D dy + dt o (Mt^T dy + e^{cs_last - cs} B G_out),
  dB = dt o (A2^T C + e^{cs_last - cs} x G_out^T),
  dC = (A2 o dt) B + e^{cs} dy h_in^T;
* d log dA_j = sum_{k >= j} dL/dcs_k, where dL/dcs_k is the row sum minus the
  column sum of W = Mt o DX o dt_j, plus e^{cs_k} dy_k . (h_in^T C_k), minus
  e^{cs_last - cs_k} dt_k x_k . (G_out^T B_k), plus <G_out, h_last> at the last
  step; ddt = x . (G^T B) + a d log dA and dA_log = a sum dt d log dA.

Each planted slip below (a dropped chain term, a sign in dL/dcs, a transposed
decay) moves some gradient far outside the bound.
"""
import numpy as np
import pytest

from oracle.backward import ssd_bwd


def _softplus(z):
    return np.maximum(z, 0) + np.log1p(np.exp(-np.abs(z)))


def chunk_bwd(x, dt_raw, dt_bias, A_log, B, C, D, init_state, dy, d_final, Q, slip=None):
    """The gradients of the scan by the chunk form above (dict as the oracle's)."""
    Bt, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    hpg = H // G
    a_all = -np.exp(A_log)
    dt_all = _softplus(dt_raw + dt_bias[None, None, :])
    out = dict(dx=np.zeros_like(x), ddt_raw=np.zeros((Bt, L, H)), dB=np.zeros((Bt, L, G, N)),
               dC=np.zeros((Bt, L, G, N)), dD=np.zeros(H), dA_log=np.zeros(H), d_init=np.zeros((Bt, H, P, N)))
    chunks = [slice(c0, min(L, c0 + Q)) for c0 in range(0, L, Q)]
    for b in range(Bt):
        for h in range(H):
            g, a = h // hpg, a_all[h]
            Bg, Cg, xh, dyh, dt = B[b, :, g], C[b, :, g], x[b, :, h], dy[b, :, h], dt_all[b, :, h]
            cs = [np.cumsum(dt[st] * a) for st in chunks]
            # the forward chain of entering states [N][P]
            h_in = [np.zeros((N, P)) if init_state is None else init_state[b, h].T.copy()]
            for k, st in enumerate(chunks[:-1]):
                w = np.exp(cs[k][-1] - cs[k]) * dt[st]
                S = (Bg[st] * w[:, None]).T @ xh[st]
                h_in.append(np.exp(cs[k][-1]) * h_in[k] + S)
            # the reverse chain of G_out [N][P]
            g_out = [None] * len(chunks)
            g_out[-1] = np.zeros((N, P)) if d_final is None else d_final[b, h].T.copy()
            for k in range(len(chunks) - 1, 0, -1):
                st = chunks[k]
                R = (Cg[st] * np.exp(cs[k])[:, None]).T @ dyh[st]
                g_out[k - 1] = np.exp(cs[k][-1]) * g_out[k] + R
            st0 = chunks[0]
            R0 = (Cg[st0] * np.exp(cs[0])[:, None]).T @ dyh[st0]
            d_init = np.exp(cs[0][-1]) * g_out[0] + R0
            if slip == "no_chain_term":
                d_init = R0
            out["d_init"][b, h] = d_init.T
            dlog_dA = np.zeros(L)
            for k, st in enumerate(chunks):
                c, Go, hi = cs[k], g_out[k], h_in[k]
                n = c.shape[0]
                Cc, Bc, xc, dyc, dtc = Cg[st], Bg[st], xh[st], dyh[st], dt[st]
                E = np.tril(np.exp(c[:, None] - c[None, :]))
                if slip == "transposed_decay":
                    E = np.tril(np.exp(c[None, :] - c[:, None]))
                CB, DX = Cc @ Bc.T, dyc @ xc.T
                Mt, A2 = E * CB, E * DX
                tail = np.exp(c[-1] - c)
                out["dx"][b, st, h] = D[h] * dyc + dtc[:, None] * (Mt.T @ dyc + tail[:, None] * (Bc @ Go))
                dBh = dtc[:, None] * (A2.T @ Cc + tail[:, None] * (xc @ Go.T))
                dCh = (A2 * dtc[None, :]) @ Bc + np.exp(c)[:, None] * (dyc @ hi.T)
                out["dB"][b, st, g] += dBh
                out["dC"][b, st, g] += dCh
                # dL/dcs_k, then d log dA by suffix sums within the chunk
                W = Mt * DX * dtc[None, :]
                dcs = W.sum(axis=1) - W.sum(axis=0)
                if slip == "sign_in_dcs":
                    dcs = W.sum(axis=1) + W.sum(axis=0)
                dcs += np.exp(c) * np.einsum("tp,np,tn->t", dyc, hi, Cc)
                dcs -= tail * dtc * np.einsum("tp,np,tn->t", xc, Go, Bc)
                h_last = np.exp(c[-1]) * hi + (Bc * (tail * dtc)[:, None]).T @ xc
                dcs[n - 1] += np.sum(Go * h_last)
                dlog = np.cumsum(dcs[::-1])[::-1]
                dlog_dA[st] = dlog
                # G_t^T B_t for ddt: G_t = sum_{s >= t} e^{cs_s - cs_t} C_s dy_s^T + tail_t G_out
                GtB = (E.T * (Cc @ Bc.T).T) @ dyc        # [t][p] = sum_s E[s,t] (C_s . B_t) dy_s
                GtB += tail[:, None] * (Bc @ Go)
                ddt = np.sum(xc * GtB, axis=1) + a * dlog
                sig = 1.0 / (1.0 + np.exp(-(dt_raw[b, st, h] + dt_bias[h])))
                out["ddt_raw"][b, st, h] = ddt * sig
            out["dA_log"][h] += a * np.sum(dt * dlog_dA)
            out["dD"][h] += np.sum(dyh * xh)
    out["ddt_bias"] = out["ddt_raw"].sum(axis=(0, 1))
    return out


def _case(seed, Bt=2, L=37, H=4, P=3, N=5, G=2, init=True, dfin=True):
    rng = np.random.default_rng(seed)
    inp = dict(x=rng.standard_normal((Bt, L, H, P)), dt_raw=0.3 * rng.standard_normal((Bt, L, H)),
               dt_bias=rng.uniform(-2.5, -0.5, H), A_log=np.log(rng.uniform(0.3, 2.0, H)),
               B=rng.standard_normal((Bt, L, G, N)), C=rng.standard_normal((Bt, L, G, N)),
               D=rng.standard_normal(H), init_state=rng.standard_normal((Bt, H, P, N)) if init else None)
    dy = rng.standard_normal((Bt, L, H, P))
    d_final = rng.standard_normal((Bt, H, P, N)) if dfin else None
    return inp, dy, d_final


def _rel(u, v):
    return float(np.max(np.abs(u - v)) / max(np.max(np.abs(v)), 1e-300))


KEYS = ("dx", "ddt_raw", "ddt_bias", "dA_log", "dB", "dC", "dD", "d_init")


@pytest.mark.parametrize("L,Q,G,init,dfin", [(37, 8, 2, True, True), (64, 16, 1, False, True),
                                             (50, 64, 2, True, False), (1, 8, 4, True, True),
                                             (33, 11, 1, True, True)])
def test_chunk_form_gradients_equal_the_oracle(L, Q, G, init, dfin):
    inp, dy, d_final = _case(L + Q + G, L=L, G=G, init=init, dfin=dfin)
    ref = ssd_bwd(**inp, dy=dy, d_final=d_final)
    got = chunk_bwd(**inp, dy=dy, d_final=d_final, Q=Q)
    for k in KEYS:
        assert _rel(got[k], ref[k]) < 1e-10, (k, _rel(got[k], ref[k]))


@pytest.mark.parametrize("slip,key", [("no_chain_term", "d_init"), ("sign_in_dcs", "dA_log"),
                                      ("transposed_decay", "dx")])
def test_planted_slips_are_caught(slip, key):
    inp, dy, d_final = _case(9, L=40)
    ref = ssd_bwd(**inp, dy=dy, d_final=d_final)
    got = chunk_bwd(**inp, dy=dy, d_final=d_final, Q=8, slip=slip)
    assert _rel(got[key], ref[key]) > 1e-3
