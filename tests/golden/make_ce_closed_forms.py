"""Writes ce_closed_forms.jsonl: small cross-entropy calls whose losses,
gradients, argmax and reduced values follow in closed form from the method's
definition ("Add Liger Kernel support for Muse Glimmer", Summary: the logits'
cross-entropy with ignore_index, label smoothing and the T tanh(x / T)
softcap; "Add Megatron-LM cross-entropy integration", Summary: mean over the
non-ignored tokens).  Python's math module only: no oracle, no GPU.

Per row with label y (not ignored), z_j = T tanh(x_j / T) (or x_j), q_j =
(1 - eps) [j = y] + eps / V:
    lse = ln sum_j exp(z_j),  loss = lse - (1 - eps) z_y - (eps / V) sum_j z_j,
    grad_j = scale (exp(z_j - lse) - q_j) (1 - tanh^2(x_j / T)),
scale = grad_scale / n_valid (mean) or grad_scale (sum); an ignored row has
loss 0 and gradient 0.  argmax = the smallest j holding max_j x_j.  Every
input value is exactly representable in bf16.  flce_closed_forms.jsonl: the
fused linear form ("Add Liger Kernel support for Muse Glimmer", Summary and
Details): logits S = h W^T of small exact inputs, then the same, with
grad_hidden = G W and grad_weight = G^T h for G = d loss / d S.

Run from this directory: python make_ce_closed_forms.py
"""
import json
import math

IGNORE = -100


def row(x, y, T, eps):
    V = len(x)
    if T > 0:
        t = [math.tanh(v / T) for v in x]
        z = [T * tv for tv in t]
        dz = [1.0 - tv * tv for tv in t]
    else:
        z = list(x)
        dz = [1.0] * V
    m = max(z)
    lse = m + math.log(math.fsum(math.exp(v - m) for v in z))
    loss = lse - (1.0 - eps) * z[y] - (eps / V) * math.fsum(z)
    p = [math.exp(v - lse) for v in z]
    return loss, p, dz


def case(name, x, labels, T=0.0, eps=0.0, reduction="mean", grad_scale=1.0, note=""):
    N, V = len(x), len(x[0])
    valid = [y != IGNORE for y in labels]
    n_valid = sum(valid)
    scale = (grad_scale / n_valid if n_valid else 0.0) if reduction == "mean" else grad_scale
    losses, grads, amax = [], [], []
    for xr, y in zip(x, labels):
        mx = max(xr)
        amax.append(min(j for j in range(V) if xr[j] == mx))
        if y == IGNORE:
            losses.append(0.0)
            grads.append([0.0] * V)
            continue
        loss, p, dz = row(xr, y, T, eps)
        q = [eps / V + ((1.0 - eps) if j == y else 0.0) for j in range(V)]
        losses.append(loss)
        grads.append([scale * (p[j] - q[j]) * dz[j] for j in range(V)])
    total = math.fsum(l for l, v in zip(losses, valid) if v)
    reduced = (total / n_valid if n_valid else 0.0) if reduction == "mean" else total
    n_correct = sum(1 for a, y, v in zip(amax, labels, valid) if v and a == y)
    accuracy = n_correct / n_valid if n_valid else 0.0
    return {"case": name, "note": note, "V": V, "softcap": T, "label_smoothing": eps,
            "reduction": reduction, "grad_scale": grad_scale, "labels": labels, "x": x,
            "loss": losses, "grad": grads, "argmax": amax, "reduced_loss": reduced,
            "accuracy": accuracy, "n_valid": n_valid, "n_correct": n_correct}


CASES = [
    case("uniform", [[0.0] * 8, [0.0] * 8], [3, IGNORE],
         note="equal logits: loss ln 8, gradient 1/8 - [j = y] over the one valid row"),
    case("two_class", [[0.0, 1.0], [1.0, 0.0]], [0, 0],
         note="two classes: loss softplus(x_1 - x_0); argmax 1 then 0"),
    case("smoothing", [[1.0, 2.0, 3.0, 4.0]], [2], eps=0.1,
         note="label smoothing 0.1: q = 0.025 + 0.9 [j = 2]"),
    case("softcap", [[-1.0, 0.5, 2.0], [4.0, -3.0, 0.25]], [1, 0], T=2.0, eps=0.2,
         reduction="sum", grad_scale=0.5,
         note="softcap T = 2 (z = 2 tanh(x / 2), dz/dx = 1 - tanh^2), sum reduction, grad_scale 0.5"),
    case("ties", [[3.0, 5.0, 5.0, 1.0], [-2.0, -2.0, -2.0, -2.0]], [2, 0],
         note="argmax ties: the smallest column (1, then 0)"),
]


def flce_case(name, h, W, labels, T=0.0, eps=0.0, reduction="mean", grad_scale=1.0, note=""):
    """The fused linear form: the logits S = h W^T (exact: small values), the
    cross-entropy of S as above with G = d loss / d S, grad_h = G W and
    grad_W = G^T h."""
    S = [[math.fsum(a * b for a, b in zip(hr, wr)) for wr in W] for hr in h]
    c = case(name, S, labels, T=T, eps=eps, reduction=reduction, grad_scale=grad_scale, note=note)
    G = c.pop("grad")
    c["S"] = c.pop("x")
    N, H, V = len(h), len(h[0]), len(W)
    c.update({"h": h, "W": W, "H": H,
              "grad_hidden": [[math.fsum(G[n][v] * W[v][k] for v in range(V)) for k in range(H)]
                              for n in range(N)],
              "grad_weight": [[math.fsum(G[n][v] * h[n][k] for n in range(N)) for k in range(H)]
                              for v in range(V)]})
    return c


def _flce_inputs(N, H, V):
    h = [[(1.0 if k == n else 0.0) + (0.5 if k == 8 else 0.0) for k in range(H)] for n in range(N)]
    W = [[float((v + k) % 3 - 1) if k < 16 else 0.0 for k in range(H)] for v in range(V)]
    return h, W


FLCE_CASES = [
    flce_case("flce_plain", *_flce_inputs(3, 64, 5), [2, 0, -100],
              note="S = h W^T with h one-hot plus 0.5 at column 8, W entries in {-1, 0, 1}"),
    flce_case("flce_softcap_smoothing", *_flce_inputs(4, 64, 7), [6, 1, 3, 0], T=2.0, eps=0.1,
              reduction="sum", grad_scale=0.5, note="softcap T = 2, smoothing 0.1, sum reduction"),
]

if __name__ == "__main__":
    with open("ce_closed_forms.jsonl", "w") as f:
        for c in CASES:
            f.write(json.dumps(c) + "\n")
    with open("flce_closed_forms.jsonl", "w") as f:
        for c in FLCE_CASES:
            f.write(json.dumps(c) + "\n")
