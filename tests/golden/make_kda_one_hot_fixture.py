"""Writes kda_one_hot_closed_form.txt: exact rationals for Phase 2 with a
per-channel decay on one-hot keys (no oracle call; closed form only).

Reading of the Kimi Delta Attention backbone named in section 4 of the
gist.science summary of "OSDN: Improving Delta Rule with Provable Online
Preconditioning in Linear Attention" (no formula printed there): the scalar
gate of the Gated DeltaNet backbone made a decay per key channel,
    S_t = S_{t-1} Diag(alpha_t) + beta_t (v_t - S_{t-1} Diag(alpha_t) k_t) ktilde_t^T.
With ktilde_t = k_t = e_{j_t} (one-hot) the key columns decouple: column
j_t takes S[:, j] <- alpha_tj (1 - beta_t) S[:, j] + beta_t v_t, every other
column j only decays, S[:, j] <- alpha_tj S[:, j].  The outputs are
o_t = S_t q_t.
"""
import os
from fractions import Fraction as F

K, V = 3, 2
S0 = [[F(1), F(-1, 2), F(0)], [F(2), F(1, 3), F(-1)]]          # [V][K]
cols = [0, 2, 0, 1, 2, 2]
beta = [F(1, 2), F(1, 3), F(3, 4), F(1), F(1, 5), F(2, 3)]
alpha = [[F(9, 10), F(1, 2), F(1)], [F(3, 4), F(1), F(4, 5)], [F(1), F(7, 8), F(1, 2)],
         [F(1, 2), F(9, 10), F(1)], [F(1), F(1), F(3, 5)], [F(5, 6), F(2, 3), F(1)]]
v = [[F(1), F(0)], [F(-1), F(2)], [F(1, 2), F(1, 2)], [F(3), F(-2)], [F(0), F(1)], [F(2), F(2)]]
q = [[F(1), F(0), F(1)], [F(0), F(1), F(0)], [F(1, 2), F(1, 2), F(1, 2)], [F(1), F(-1), F(0)],
     [F(0), F(0), F(1)], [F(1), F(2), F(3)]]

S = [row[:] for row in S0]
o = []
for t, j in enumerate(cols):
    for i in range(V):
        for c in range(K):
            if c == j:
                S[i][c] = alpha[t][c] * (1 - beta[t]) * S[i][c] + beta[t] * v[t][i]
            else:
                S[i][c] = alpha[t][c] * S[i][c]
    o.append([sum(S[i][c] * q[t][c] for c in range(K)) for i in range(V)])

out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "kda_one_hot_closed_form.txt")
line = lambda xs: " ".join(str(x) for x in xs)
with open(out, "w") as f:
    f.write("# Phase 2 with a per-channel decay on one-hot keys, exact rationals.\n")
    f.write("# Key column j_t: alpha (1 - beta) S + beta v; other columns: alpha S.\n")
    f.write("# Written by make_kda_one_hot_fixture.py.\n")
    f.write("K = %d\nV = %d\n" % (K, V))
    f.write("cols = %s\n" % line(cols))
    f.write("beta = %s\n" % line(beta))
    for t in range(len(cols)):
        f.write("alpha_%d = %s\n" % (t, line(alpha[t])))
        f.write("v_%d = %s\n" % (t, line(v[t])))
        f.write("q_%d = %s\n" % (t, line(q[t])))
    for i in range(V):
        f.write("S0_%d = %s\n" % (i, line(S0[i])))
    for t in range(len(cols)):
        f.write("o_%d = %s\n" % (t, line(o[t])))
    for i in range(V):
        f.write("ST_%d = %s\n" % (i, line(S[i])))
