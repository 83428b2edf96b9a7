"""CPU fp64 oracle for the fused linear cross-entropy (FLCE) of a language-model head.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline leg may import or run this module. It shares no code with the CUDA
path and never takes an input or an expected value from it.

What it computes, read from the pages:

* Liger-Kernel, "Muse Glimmer" support, section Summary item 1: the loss of the
  LM head without keeping a [batch, seq, vocab] logits tensor around. The
  oracle does keep logits, one block of at most `block_rows` rows at a time,
  in fp64: that is the plain definition the fused path must reproduce.
* Same page, section Details / Softcap: HF caps as T*tanh(logits*m/T); the
  output multiplier m is folded into the hidden states since
  (m*h) W^T = m (h W^T). The oracle scales h by m (fp64, exact) and then caps.
* Same page, Summary item 2 and Testing Done: token_accuracy and
  predicted_tokens come out of the fused path.
* Liger-Kernel, DeepSeek-V3 support, section Memory, and the Muse Glimmer page,
  section Memory: grad_weight is accumulated in fp32; here the caller's
  accumulator G0 is added to (G0 + dL/dW), in fp64.
* SpecForge DSpine PR, section Changes: a frozen vocabulary projection has no
  weight gradient (need_grad_W=False).

Readings where the pages are silent: the loss is the mean over rows whose label
is not ignore_index (n_valid); n_valid = 0 gives loss 0, accuracy 0 and zero
gradients; argmax ties go to the lowest vocab index; predicted tokens are
reported for every row, ignored or not; the argmax is taken on the capped
logits; T = 0 means no softcap; grad_scale g multiplies every gradient.

Definition, per row i (all in fp64):
    z_i   = (m h_i) W^T                                  [V]
    s_i   = T tanh(z_i / T)   if T > 0, else z_i
    lse_i = max_j s_ij + log sum_j exp(s_ij - max_j s_ij)
    l_i   = lse_i - s_{i, y_i}                            (valid rows)
    loss  = sum_valid l_i / n_valid   (mean)   or   sum_valid l_i   (sum)
    pred_i = min { j : s_ij = max_j s_ij }
    acc   = #{valid i : pred_i = y_i} / n_valid
    q_ij  = c (softmax(s_i)_j - [j = y_i]),   c = g / n_valid (mean) or g (sum),
            q_ij = 0 on ignored rows
    dz_ij = q_ij (1 - (s_ij / T)^2)   if T > 0, else q_ij
    grad_h_i = m sum_j dz_ij W_j
    grad_W_j = G0_j + sum_i dz_ij (m h_i)
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "capped_logits",
    "flce_oracle",
    "oracle_rows",
    "oracle_grad_W_rows",
    "oracle_ce_logits",
    "oracle_shard_partials",
    "oracle_merge_shards",
    "oracle_shard_grad_h",
]


def _f64(x) -> np.ndarray:
    """fp64 view of an array-like (torch tensors are converted through fp32,
    which holds every bf16 value exactly)."""
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if x.dtype.is_floating_point:
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def _i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.asarray(x, dtype=np.int64)


def capped_logits(h_rows: np.ndarray, W: np.ndarray, softcap: float, out_mult: float):
    """z = (m h) W^T and s = softcap(z) for a block of rows (Muse Glimmer page,
    Details / Softcap: m is folded into h, then T tanh(z / T))."""
    hm = out_mult * h_rows
    z = hm @ W.T
    if softcap > 0.0:
        s = softcap * np.tanh(z / softcap)
    else:
        s = z
    return z, s


def _coef(n_valid: int, reduction: str, grad_scale: float) -> float:
    if n_valid == 0:
        return 0.0
    if reduction == "mean":
        return grad_scale / n_valid
    if reduction == "sum":
        return grad_scale
    raise ValueError(f"unknown reduction {reduction!r}")


def _row_stats(s: np.ndarray, lab: np.ndarray, valid: np.ndarray):
    """Per-row lse, argmax (lowest index on ties), top-2 relative gap, row loss."""
    mx = s.max(axis=1)
    lse = mx + np.log(np.exp(s - mx[:, None]).sum(axis=1))
    pred = s.argmax(axis=1).astype(np.int64)          # first maximum = lowest index
    if s.shape[1] >= 2:
        second = np.partition(s, s.shape[1] - 2, axis=1)[:, -2]
        gap = (mx - second) / np.maximum(np.abs(mx), 1e-300)
    else:
        gap = np.full(s.shape[0], np.inf)
    row_loss = np.zeros(s.shape[0])
    vi = np.nonzero(valid)[0]
    row_loss[vi] = lse[vi] - s[vi, lab[vi]]
    return lse, pred, gap, row_loss


def _dz(s: np.ndarray, lse: np.ndarray, lab: np.ndarray, valid: np.ndarray,
        coef: float, softcap: float) -> np.ndarray:
    p = np.exp(s - lse[:, None])
    q = p
    vi = np.nonzero(valid)[0]
    q[vi, lab[vi]] -= 1.0
    q *= coef
    q[~valid] = 0.0
    if softcap > 0.0:
        q = q * (1.0 - (s / softcap) ** 2)
    return q


def flce_oracle(h, W, labels, *, softcap: float = 0.0, out_mult: float = 1.0,
                ignore_index: int = -100, reduction: str = "mean", grad_scale: float = 1.0,
                grad_W0=None, need_grad_h: bool = True, need_grad_W: bool = True,
                block_rows: int = 256) -> dict:
    """Full oracle: every output of the fused path for all rows.

    h [N, H], W [V, H], labels [N] (int, ignore_index marks ignored rows).
    Labels outside {ignore_index} U [0, V) raise ValueError (the fused path
    reports them as an error status).
    Returns a dict: loss, token_accuracy, n_valid, correct, predicted [N],
    lse [N], row_loss [N], top2_gap [N], and grad_h [N, H] / grad_W [V, H]
    when asked for (grad_W includes G0 when grad_W0 is given).
    """
    h = _f64(h)
    W = _f64(W)
    lab = _i64(labels)
    N, H = h.shape
    V = W.shape[0]
    valid = lab != ignore_index
    if np.any((lab[valid] < 0) | (lab[valid] >= V)):
        raise ValueError("label outside [0, V) that is not ignore_index")
    n_valid = int(valid.sum())
    coef = _coef(n_valid, reduction, grad_scale)

    lse = np.zeros(N)
    pred = np.zeros(N, dtype=np.int64)
    gap = np.zeros(N)
    row_loss = np.zeros(N)
    grad_h = np.zeros((N, H)) if need_grad_h else None
    if need_grad_W:
        grad_W = np.zeros((V, H)) if grad_W0 is None else _f64(grad_W0).copy()
    else:
        grad_W = None

    for r0 in range(0, N, block_rows):
        r1 = min(N, r0 + block_rows)
        lb = np.where(valid[r0:r1], lab[r0:r1], 0)
        vb = valid[r0:r1]
        _, s = capped_logits(h[r0:r1], W, softcap, out_mult)
        lse[r0:r1], pred[r0:r1], gap[r0:r1], row_loss[r0:r1] = _row_stats(s, lb, vb)
        if need_grad_h or need_grad_W:
            dz = _dz(s, lse[r0:r1], lb, vb, coef, softcap)
            if need_grad_h:
                grad_h[r0:r1] = out_mult * (dz @ W)
            if need_grad_W:
                grad_W += dz.T @ (out_mult * h[r0:r1])

    total = float(row_loss[valid].sum())
    correct = int(np.sum(valid & (pred == lab)))
    if n_valid == 0:
        loss, acc = 0.0, 0.0
    else:
        loss = total / n_valid if reduction == "mean" else total
        acc = correct / n_valid
    return {
        "loss": loss, "token_accuracy": acc, "n_valid": n_valid, "correct": correct,
        "predicted": pred, "lse": lse, "row_loss": row_loss, "top2_gap": gap,
        "grad_h": grad_h, "grad_W": grad_W,
    }


def oracle_rows(h_rows, W, labels_rows, n_valid: int, *, softcap: float = 0.0,
                out_mult: float = 1.0, ignore_index: int = -100, reduction: str = "mean",
                grad_scale: float = 1.0, need_grad_h: bool = True, block_rows: int = 256) -> dict:
    """Per-row outputs for a subset of rows, given the batch's n_valid.

    Row i's lse, argmax, loss term and grad_h row depend on row i alone and on
    the batch-wide n_valid (through the mean), so a sample of rows can be
    checked one by one on a head of any size.
    """
    h = _f64(h_rows)
    W = _f64(W)
    lab = _i64(labels_rows)
    R, H = h.shape
    V = W.shape[0]
    valid = lab != ignore_index
    coef = _coef(n_valid, reduction, grad_scale)
    lse = np.zeros(R)
    pred = np.zeros(R, dtype=np.int64)
    gap = np.zeros(R)
    row_loss = np.zeros(R)
    grad_h = np.zeros((R, H)) if need_grad_h else None
    for r0 in range(0, R, block_rows):
        r1 = min(R, r0 + block_rows)
        lb = np.where(valid[r0:r1], lab[r0:r1], 0)
        vb = valid[r0:r1]
        _, s = capped_logits(h[r0:r1], W, softcap, out_mult)
        lse[r0:r1], pred[r0:r1], gap[r0:r1], row_loss[r0:r1] = _row_stats(s, lb, vb)
        if need_grad_h:
            dz = _dz(s, lse[r0:r1], lb, vb, coef, softcap)
            grad_h[r0:r1] = out_mult * (dz @ W)
    return {"lse": lse, "predicted": pred, "top2_gap": gap, "row_loss": row_loss,
            "grad_h": grad_h}


def oracle_grad_W_rows(h, W, labels, vocab_ids, lse, n_valid: int, *, softcap: float = 0.0,
                       out_mult: float = 1.0, ignore_index: int = -100,
                       reduction: str = "mean", grad_scale: float = 1.0,
                       block_rows: int = 4096) -> np.ndarray:
    """dL/dW for the listed vocab rows only (without G0), given every row's lse
    from this oracle: grad_W_j = sum_i dz_ij (m h_i) needs column j of the
    logits for all rows, and each row's lse."""
    h = _f64(h)
    W = _f64(W)
    lab = _i64(labels)
    ids = _i64(vocab_ids)
    lse = _f64(lse)
    N, H = h.shape
    valid = lab != ignore_index
    coef = _coef(n_valid, reduction, grad_scale)
    out = np.zeros((ids.shape[0], H))
    Wj = W[ids]
    for r0 in range(0, N, block_rows):
        r1 = min(N, r0 + block_rows)
        hm = out_mult * h[r0:r1]
        z = hm @ Wj.T                                    # [R, k]
        s = softcap * np.tanh(z / softcap) if softcap > 0.0 else z
        p = np.exp(s - lse[r0:r1, None])
        q = p
        lb = lab[r0:r1]
        vb = valid[r0:r1]
        q -= (lb[:, None] == ids[None, :]) & vb[:, None]
        q *= coef
        q[~vb] = 0.0
        if softcap > 0.0:
            q = q * (1.0 - (s / softcap) ** 2)
        out += q.T @ hm
    return out


def oracle_ce_logits(logits, labels, *, softcap: float = 0.0, out_mult: float = 1.0,
                     ignore_index: int = -100, reduction: str = "mean", grad_scale: float = 1.0,
                     row_scale=None, need_grad: bool = True, block_rows: int = 256) -> dict:
    """Cross-entropy on logits that are already materialised: the non-fused
    branch the Muse Glimmer page tests next to the fused path (Testing Done:
    "the non-fused softcap branch"; Details: HF caps T tanh(logits m / T)), and
    the path DeepSeek-V3's lce_forward takes when logits are kept (Summary).

    Same row definition as flce_oracle with z = m * logits:
        s = T tanh(z / T) (T > 0) or z;  l_i = lse_i - s_{i, y_i}
    reduction "mean" / "sum" as there; "none" returns the row losses only
    (loss = their sum) and takes its upstream gradient per row from row_scale
    (default all ones): q_ij = row_scale_i (softmax - onehot) on valid rows.
    grad_logits = dL/dlogits = m * dz, dz as in flce_oracle.
    """
    x = _f64(logits)
    lab = _i64(labels)
    N, V = x.shape
    valid = lab != ignore_index
    if np.any((lab[valid] < 0) | (lab[valid] >= V)):
        raise ValueError("label outside [0, V) that is not ignore_index")
    n_valid = int(valid.sum())
    rs = np.ones(N) if row_scale is None else _f64(row_scale)
    lse = np.zeros(N)
    pred = np.zeros(N, dtype=np.int64)
    gap = np.zeros(N)
    row_loss = np.zeros(N)
    grad = np.zeros((N, V)) if need_grad else None
    for r0 in range(0, N, block_rows):
        r1 = min(N, r0 + block_rows)
        z = out_mult * x[r0:r1]
        s = softcap * np.tanh(z / softcap) if softcap > 0.0 else z
        lb = np.where(valid[r0:r1], lab[r0:r1], 0)
        vb = valid[r0:r1]
        lse[r0:r1], pred[r0:r1], gap[r0:r1], row_loss[r0:r1] = _row_stats(s, lb, vb)
        if need_grad:
            if reduction == "none":
                dz = _dz(s, lse[r0:r1], lb, vb, 1.0, softcap) * rs[r0:r1, None]
            else:
                dz = _dz(s, lse[r0:r1], lb, vb, _coef(n_valid, reduction, grad_scale), softcap)
            grad[r0:r1] = out_mult * dz
    total = float(row_loss[valid].sum())
    correct = int(np.sum(valid & (pred == lab)))
    if n_valid == 0:
        loss, acc = 0.0, 0.0
    else:
        loss = total / n_valid if reduction == "mean" else total
        acc = correct / n_valid
    return {"loss": loss, "token_accuracy": acc, "n_valid": n_valid, "correct": correct,
            "predicted": pred, "lse": lse, "row_loss": row_loss, "top2_gap": gap, "grad_logits": grad}


def oracle_shard_partials(h, W, labels, offsets, *, softcap: float = 0.0, out_mult: float = 1.0,
                          ignore_index: int = -100, block_rows: int = 256) -> dict:
    """Per-row partials of each vocabulary shard of W, the quantities a
    vocabulary-sharded head exchanges (the distributed DDP / FSDP runs of the
    SpecForge DSpine PR, section Validation, split W by vocabulary rows).

    offsets: S + 1 increasing vocab ids from 0 to V; shard k holds W's rows
    [offsets[k], offsets[k+1]). For each shard k and row i, over j in the shard:
        max[k, i]    = max_j s_ij
        sumexp[k, i] = sum_j exp(s_ij - max[k, i])
        argmax[k, i] = min { j : s_ij = max[k, i] }   (a global vocab id)
        target[k, i] = s_{i, y_i} if y_i is in the shard, else 0
    with s the capped logits of flce_oracle.
    """
    h = _f64(h)
    W = _f64(W)
    lab = _i64(labels)
    off = [int(o) for o in offsets]
    N = h.shape[0]
    S = len(off) - 1
    out = {k: np.zeros((S, N)) for k in ("max", "sumexp", "target")}
    out["argmax"] = np.zeros((S, N), dtype=np.int64)
    for r0 in range(0, N, block_rows):
        r1 = min(N, r0 + block_rows)
        _, s = capped_logits(h[r0:r1], W, softcap, out_mult)
        for k in range(S):
            sk = s[:, off[k]:off[k + 1]]
            mk = sk.max(axis=1)
            out["max"][k, r0:r1] = mk
            out["sumexp"][k, r0:r1] = np.exp(sk - mk[:, None]).sum(axis=1)
            out["argmax"][k, r0:r1] = off[k] + sk.argmax(axis=1)
            for i in range(r0, r1):
                y = lab[i]
                if y != ignore_index and off[k] <= y < off[k + 1]:
                    out["target"][k, i] = s[i - r0, y]
    return out


def oracle_merge_shards(part: dict, labels, offsets, *, ignore_index: int = -100, reduction: str = "mean") -> dict:
    """The batch outputs from every shard's partials (oracle_shard_partials):
        M_i    = max_k max[k, i]
        lse_i  = M_i + log sum_k sumexp[k, i] exp(max[k, i] - M_i)
        pred_i = argmax[k*, i], k* the first (lowest-id) shard with max[k*, i] = M_i
        l_i    = lse_i - target[k(y_i), i], k(y_i) the shard holding the label
    and the loss and accuracy over the valid rows as in flce_oracle."""
    lab = _i64(labels)
    off = [int(o) for o in offsets]
    mx = np.asarray(part["max"])
    S, N = mx.shape
    M = mx.max(axis=0)
    lse = M + np.log((np.asarray(part["sumexp"]) * np.exp(mx - M[None, :])).sum(axis=0))
    first = np.argmax(mx == M[None, :], axis=0)
    pred = np.asarray(part["argmax"])[first, np.arange(N)]
    valid = lab != ignore_index
    row_loss = np.zeros(N)
    for i in np.nonzero(valid)[0]:
        k = max(kk for kk in range(S) if off[kk] <= lab[i])
        row_loss[i] = lse[i] - part["target"][k][i]
    n_valid = int(valid.sum())
    correct = int(np.sum(valid & (pred == lab)))
    total = float(row_loss[valid].sum())
    if n_valid == 0:
        loss, acc = 0.0, 0.0
    else:
        loss = total / n_valid if reduction == "mean" else total
        acc = correct / n_valid
    return {"loss": loss, "token_accuracy": acc, "n_valid": n_valid, "correct": correct, "predicted": pred,
            "lse": lse, "row_loss": row_loss}


def oracle_shard_grad_h(h, W, labels, lse, n_valid: int, v0: int, v1: int, *, softcap: float = 0.0,
                        out_mult: float = 1.0, ignore_index: int = -100, reduction: str = "mean",
                        grad_scale: float = 1.0, block_rows: int = 256) -> np.ndarray:
    """One vocabulary shard's part of grad_h: m sum_{j in [v0, v1)} dz_ij W_j,
    with dz as in flce_oracle from every row's full lse. Summed over shards
    that tile [0, V) it is flce_oracle's grad_h."""
    h = _f64(h)
    W = _f64(W)
    lab = _i64(labels)
    lse = _f64(lse)
    N, H = h.shape
    valid = lab != ignore_index
    coef = _coef(n_valid, reduction, grad_scale)
    Wk = W[v0:v1]
    out = np.zeros((N, H))
    for r0 in range(0, N, block_rows):
        r1 = min(N, r0 + block_rows)
        _, s = capped_logits(h[r0:r1], Wk, softcap, out_mult)
        q = np.exp(s - lse[r0:r1, None])
        lb = lab[r0:r1]
        vb = valid[r0:r1]
        for i in range(r1 - r0):
            if vb[i] and v0 <= lb[i] < v1:
                q[i, lb[i] - v0] -= 1.0
        q *= coef
        q[~vb] = 0.0
        if softcap > 0.0:
            q = q * (1.0 - (s / softcap) ** 2)
        out[r0:r1] = out_mult * (q @ Wk)
    return out
