"""Writes one_hot_apf_closed_form.txt: exact rationals for the preconditioner
scan on one-hot keys (no oracle call; closed form only).

With a one-hot key e_i the pages' quantities reduce to ||k||^2 = 1 and
<d, k^2> = d_i (gist.science summary, section 2.2), so one APF step
(section 2.3, descent reading) touches coordinate i as
    d_i <- (r - eta beta^2) d_i + eta beta
and only rescales the others, d_j <- r d_j.
"""
import os
from fractions import Fraction as F

K = 3
beta, eta = F(1, 2), F(1, 5)
d0 = [F(1), F(2), F(1, 2)]
hits = [0, 1, 0, 2, 0, 0, 1, 2, 2, 0]
r = [F(9, 10), F(4, 5), F(1), F(3, 4), F(9, 10), F(1), F(7, 8), F(1), F(19, 20), F(2, 3)]

d = list(d0)
for i, rt in zip(hits, r):
    d = [(rt - eta * beta * beta) * dj + eta * beta if j == i else rt * dj
         for j, dj in enumerate(d)]

out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "one_hot_apf_closed_form.txt")
with open(out, "w") as f:
    f.write("# One-hot keys through the OSDN preconditioner scan, exact rationals.\n")
    f.write("# Closed form of the section 2.2/2.3 update for k_t = e_i (gist.science\n")
    f.write("# summary of arXiv 2605.13473): d_i <- (r - eta beta^2) d_i + eta beta,\n")
    f.write("# d_j <- r d_j (j != i).  Written by make_one_hot_fixture.py.\n")
    f.write("K = %d\nbeta = %s\neta = %s\n" % (K, beta, eta))
    f.write("d0 = %s\n" % " ".join(str(x) for x in d0))
    f.write("hits = %s\n" % " ".join(str(x) for x in hits))
    f.write("r = %s\n" % " ".join(str(x) for x in r))
    f.write("dT = %s\n" % " ".join(str(x) for x in d))
