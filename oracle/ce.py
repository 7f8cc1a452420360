"""Cross-entropy over the LM head, loss and dH -- oracle (test infrastructure only).

"Exact Layer Streaming ..." (abstract) singles out the cross-entropy logits
term as a measured memory cost (14 bytes per logit element against 6 from
first principles); the library's job is the same loss with the logits never
held in full.  What is computed is the plain definition:

    z_i   = W h_i                         (W [V, D] head, h_i a row of H [M, D])
    lse_i = log sum_v exp(z_iv)
    loss  = (1/N_valid) sum_{i valid} (lse_i - z_{i,label_i})
    dH_i  = (softmax(z_i) - onehot(label_i)) W / N_valid   for valid rows, 0 otherwise

Readings (the pages are silent): labels are already aligned with rows (no
shift inside the call); a row whose label equals ``ignore_index`` (-100)
contributes nothing; with N_valid == 0 the loss and dH are 0 (not NaN).
Float64 throughout, rows processed in chunks only to bound memory.
"""
import numpy as np


def ce_rows(H, W, labels, n_valid, ignore_index=-100, want_soft=False, want_grad=True):
    """Per-row loss terms and dH rows for the given rows, with the global N_valid.

    want_grad=False skips the dH rows (loss terms only); it changes no value.
    """
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64) if np.asarray(W).dtype != np.float64 else W
    labels = np.asarray(labels)
    M = H.shape[0]
    terms = np.zeros(M)
    dH = np.zeros_like(H)
    soft = np.zeros_like(H) if want_soft else None
    if n_valid == 0:
        return terms, dH, soft
    for s in range(0, M, 64):
        Z = H[s:s + 64] @ W.T
        zmax = Z.max(axis=1, keepdims=True)
        lse = zmax[:, 0] + np.log(np.exp(Z - zmax).sum(axis=1))
        P = np.exp(Z - lse[:, None])
        lab = labels[s:s + 64]
        valid = lab != ignore_index
        idx = np.nonzero(valid)[0]
        terms[s + idx] = lse[idx] - Z[idx, lab[idx]]
        P[~valid] = 0.0
        if not want_grad:
            continue
        if want_soft:
            soft[s:s + 64] = (P @ W) / n_valid
        P[idx, lab[idx]] -= 1.0
        dH[s:s + 64] = (P @ W) / n_valid
    return terms, dH, soft


def ce_fwd_bwd(H, W, labels, ignore_index=-100, want_soft=False):
    """(loss, dH[, softmax part of dH]) of the mean cross-entropy over valid rows."""
    labels = np.asarray(labels)
    n_valid = int(np.sum(labels != ignore_index))
    W64 = np.asarray(W, dtype=np.float64)
    terms, dH, soft = ce_rows(H, W64, labels, n_valid, ignore_index, want_soft)
    loss = float(terms.sum() / n_valid) if n_valid else 0.0
    return (loss, dH, soft) if want_soft else (loss, dH)
