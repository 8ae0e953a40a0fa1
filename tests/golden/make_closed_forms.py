"""Writes tests/golden/closed_forms.json: 4x4 cases whose Birkhoff projection
(and, for one case, whose backward pass) is known in closed form.

The pages print no worked example, so the fixtures are closed forms of the
definition they give: P is the unique doubly stochastic matrix of the form
diag(e^a) exp(X) diag(e^b) ("Accelerating the Birkhoff Projection for
Manifold-Constrained Hyper-Connections", s1 and s2: projection onto the
Birkhoff polytope as entropic optimal transport).  Each case states its
derivation.  Values are computed here with exact rational arithmetic (and
math.log for the logits); nothing is computed by the CUDA library or by the
oracle.

Run:  python tests/golden/make_closed_forms.py
"""
import json
import math
import os
from fractions import Fraction as F

HERE = os.path.dirname(os.path.abspath(__file__))


def fl(m):
    return [[float(v) for v in row] for row in m]


def perm_matrix(perm):
    return [[F(1) if perm[i] == j else F(0) for j in range(4)] for i in range(4)]


cases = []

# 1. X = 0: exp(X) is the all-ones matrix, already a scaled doubly stochastic
#    matrix; P = J/4.
cases.append(dict(
    name="zeros",
    derivation="exp(0) = J; J/4 is doubly stochastic and of the form D1 J D2, so P = J/4",
    X=fl([[0] * 4] * 4), P=fl([[F(1, 4)] * 4] * 4)))

# 2. X_ij = u_i + v_j: exp(X) = diag(e^u) J diag(e^v), so again P = J/4.
u = [1.0, -2.0, 3.0, 0.5]
v = [0.0, 7.0, -3.0, 2.0]
cases.append(dict(
    name="rank_one_offsets",
    derivation="X = u 1^T + 1 v^T makes exp(X) = diag(e^u) J diag(e^v); P = J/4",
    X=[[u[i] + v[j] for j in range(4)] for i in range(4)], P=fl([[F(1, 4)] * 4] * 4)))

# 3. X = c I with c = ln 3: by symmetry P = alpha I + beta (J - I) with
#    alpha = e^c beta and (e^c + 3) beta = 1: alpha = 1/2, beta = 1/6.
c = math.log(3.0)
cases.append(dict(
    name="diag_ln3",
    derivation="X = cI: P_ii = e^c/(e^c+3), P_ij = 1/(e^c+3); c = ln 3 gives 1/2 and 1/6",
    X=[[c if i == j else 0.0 for j in range(4)] for i in range(4)],
    P=fl([[F(1, 2) if i == j else F(1, 6) for j in range(4)] for i in range(4)])))

# 4. X = c I with c = -ln 2: alpha = (1/2)/(1/2 + 3) = 1/7, beta = 2/7.
c = -math.log(2.0)
cases.append(dict(
    name="diag_minus_ln2",
    derivation="X = cI with c = -ln 2: P_ii = (1/2)/(7/2) = 1/7, P_ij = 2/7",
    X=[[c if i == j else 0.0 for j in range(4)] for i in range(4)],
    P=fl([[F(1, 7) if i == j else F(2, 7) for j in range(4)] for i in range(4)])))

# 5. Circulant X_ij = x_{(j-i) mod 4} with e^x = (1, 2, 3, 4): every row of the
#    row softmax is a cyclic shift of (1,2,3,4)/10 and every column holds each
#    value once, so the row softmax is already doubly stochastic.
w = [F(1, 10), F(2, 10), F(3, 10), F(4, 10)]
x = [math.log(1.0), math.log(2.0), math.log(3.0), math.log(4.0)]
cases.append(dict(
    name="circulant",
    derivation="circulant logits: the row softmax has unit column sums, so P = rowsoftmax(X)",
    X=[[x[(j - i) % 4] for j in range(4)] for i in range(4)],
    P=fl([[w[(j - i) % 4] for j in range(4)] for i in range(4)])))

# 6. Fixed point: Q = 0.4 I + 0.3 Pi1 + 0.2 Pi2 + 0.1 Pi3 (Klein four-group
#    permutations) is strictly positive and doubly stochastic; for
#    X = log Q + u 1^T + 1 v^T uniqueness gives P = Q.
Q = [[F(0)] * 4 for _ in range(4)]
for wgt, perm in ((F(4, 10), (0, 1, 2, 3)), (F(3, 10), (1, 0, 3, 2)),
                  (F(2, 10), (2, 3, 0, 1)), (F(1, 10), (3, 2, 1, 0))):
    pm = perm_matrix(perm)
    for i in range(4):
        for j in range(4):
            Q[i][j] += wgt * pm[i][j]
uu = [3.0, -1.0, 0.5, 2.0]
vv = [-4.0, 0.0, 1.5, 10.0]
cases.append(dict(
    name="fixed_point_klein",
    derivation="X = log Q + u 1^T + 1 v^T with Q doubly stochastic and positive: P = Q",
    X=[[math.log(float(Q[i][j])) + uu[i] + vv[j] for j in range(4)] for i in range(4)],
    P=fl(Q)))

# Backward at X = 0 (P = J/4): with r = row means R_i of G, c = column means
# C_j, y = c - P^T r = C - mean(G); the dual Hessian is I - J/4, whose reduced
# solve gives beta_j = y_j - y_3 and alpha_i = R_i + y_3, hence
#   dX = P o (G - alpha 1^T - 1 beta^T) = (G_ij - R_i - C_j + mean(G)) / 4.
G = [[F(1), F(2), F(3), F(4)],
     [F(0), F(-1), F(5), F(2)],
     [F(3), F(3), F(-2), F(0)],
     [F(1), F(0), F(0), F(7)]]
R = [sum(G[i]) / 4 for i in range(4)]
C = [sum(G[i][j] for i in range(4)) / 4 for j in range(4)]
Gm = sum(sum(r) for r in G) / 16
dX = [[(G[i][j] - R[i] - C[j] + Gm) / 4 for j in range(4)] for i in range(4)]
backward_cases = [dict(
    name="zeros_backward",
    derivation="at X = 0: dX = (G - row means - column means + grand mean) / 4",
    X=fl([[0] * 4] * 4), G=fl(G), dX=fl(dX))]

out = dict(
    source=("Accelerating the Birkhoff Projection for Manifold-Constrained "
            "Hyper-Connections, s1-s2.2 (definition of the projection and of "
            "its implicit-differentiation backward); values are closed forms"),
    forward=cases, backward=backward_cases)


def dump(obj, ind=0):
    # compact JSON: one matrix row per line
    pad = " " * ind
    if isinstance(obj, dict):
        items = [pad + " " + json.dumps(k) + ": " + dump(v, ind + 1).lstrip() for k, v in obj.items()]
        return pad + "{\n" + ",\n".join(items) + "\n" + pad + "}"
    if isinstance(obj, list) and obj and isinstance(obj[0], list) and not isinstance(obj[0][0], (list, dict)):
        return pad + "[" + (",\n" + pad + " ").join(json.dumps(r) for r in obj) + "]"
    if isinstance(obj, list):
        return pad + "[\n" + ",\n".join(dump(v, ind + 1) for v in obj) + "\n" + pad + "]"
    return pad + json.dumps(obj)


with open(os.path.join(HERE, "closed_forms.json"), "w") as f:
    f.write(dump(out) + "\n")
print("wrote", len(cases), "forward and", len(backward_cases), "backward cases")
