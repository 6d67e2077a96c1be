"""Selection-quality measurement (paper summary page "Block Sparse Attention with
Log-Linear Complexity", section "Experimental results", item 4 and Figure 2: Recall@K of
the selected blocks against the full-attention reference blocks, and the attention mass
the selection keeps, by query position).

This is measurement code, not part of the selection or attention path: it recomputes, for
a sample of queries, the exact leaf-level block scores over every eligible block (the LSE
of each block's raw-key logits summed over the group's heads, i.e. what the method would
rank if nothing were pruned) and dense causal attention, with plain PyTorch on whatever
device the tensors are on.

Readings: the reference set of a query is the top-K of those exact scores with the query's
own block always kept and ties to the lower block index, the same rule as the method's
final top-K; Recall@K = |selected ∩ reference| / |reference|.  The kept mass of a query head
is the sum of its dense softmax weights over the keys of the selected blocks (keys <= t).
"""
from __future__ import annotations

import math

import torch


def _block_lse(logits: torch.Tensor, C: int) -> torch.Tensor:
    """logits [..., n] (masked entries -inf) -> per-block LSE [..., ceil(n / C)]."""
    n = logits.shape[-1]
    m = -(-n // C)
    pad = m * C - n
    if pad:
        logits = torch.nn.functional.pad(logits, (0, pad), value=-math.inf)
    return torch.logsumexp(logits.reshape(*logits.shape[:-1], m, C), dim=-1)


def exact_topk_blocks(Q, K, b: int, t: int, K_sel: int, C: int = 64, scale: float | None = None) -> torch.Tensor:
    """Reference block set [H_kv, K_sel] (ascending, -1 padded) for causal query (b, t).
    Q [B, N, H_q, d], K [B, H_kv, N_cap, d] (bf16 or float)."""
    H_q, d = Q.shape[2], Q.shape[3]
    H_kv = K.shape[1]
    G = H_q // H_kv
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    q = Q[b, t].double().reshape(H_kv, G, d)
    k = K[b, :, : t + 1].double()                                   # [H_kv, t+1, d]
    logits = scale * torch.einsum("hgd,hnd->hgn", q, k)             # [H_kv, G, t+1]
    score = _block_lse(logits, C).sum(dim=1)                        # [H_kv, blocks]
    own = t // C
    out = torch.full((H_kv, K_sel), -1, dtype=torch.int64)
    for h in range(H_kv):
        s = score[h].clone()
        s[own] = -math.inf
        order = torch.sort(s, descending=True, stable=True).indices   # ties: lower index first
        keep = [int(j) for j in order[: K_sel - 1].tolist() if s[j] > -math.inf]
        blocks = sorted(keep + [own])
        out[h, : len(blocks)] = torch.tensor(blocks)
    return out


def kept_attention_mass(Q, K, idx_row, b: int, t: int, C: int = 64, scale: float | None = None) -> torch.Tensor:
    """Dense causal softmax mass of query (b, t) on the keys of its selected blocks:
    idx_row [H_kv, K_sel] -> [H_q]."""
    H_q, d = Q.shape[2], Q.shape[3]
    H_kv = K.shape[1]
    G = H_q // H_kv
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    q = Q[b, t].double().reshape(H_kv, G, d)
    k = K[b, :, : t + 1].double()
    w = torch.softmax(scale * torch.einsum("hgd,hnd->hgn", q, k), dim=-1)   # [H_kv, G, t+1]
    blk = torch.arange(t + 1, device=w.device) // C
    mass = torch.zeros(H_kv, G, dtype=torch.float64, device=w.device)
    for h in range(H_kv):
        sel = idx_row[h][idx_row[h] >= 0].to(w.device)
        mask = torch.isin(blk, sel)
        mass[h] = w[h][:, mask].sum(dim=-1)
    return mass.reshape(H_q)


def selection_quality(Q, K, idx, K_sel: int, rows, C: int = 64, scale: float | None = None, buckets: int = 4) -> dict:
    """idx [B, H_kv, N, K_sel] from the selection under test; rows: iterable of (b, t).
    Returns mean Recall@K and kept mass overall and per query-position bucket."""
    N = Q.shape[1]
    rec, mass, pos = [], [], []
    for b, t in rows:
        ref = exact_topk_blocks(Q, K, b, t, K_sel, C, scale)
        got = idx[b, :, t].to("cpu", torch.int64)
        for h in range(ref.shape[0]):
            r = set(ref[h][ref[h] >= 0].tolist())
            g = set(got[h][got[h] >= 0].tolist())
            rec.append(len(r & g) / max(1, len(r)))
            pos.append(t)
        mass.append(kept_attention_mass(Q, K, got, b, t, C, scale).mean().item())
    rec_t = torch.tensor(rec)
    pos_t = torch.tensor(pos)
    out = {"recall_at_k": float(rec_t.mean()), "kept_mass": float(torch.tensor(mass).mean()), "queries": len(mass)}
    edges = [N * i // buckets for i in range(buckets + 1)]
    out["recall_by_position"] = [float(rec_t[(pos_t >= lo) & (pos_t < hi)].mean()) if ((pos_t >= lo) & (pos_t < hi)).any()
                                 else None for lo, hi in zip(edges[:-1], edges[1:])]
    return out


def needle_hit_rate(idx, targets, C: int = 64) -> dict:
    """Share of planted-needle query rows whose selected set holds the needle's block.

    idx [B, H_kv, N, K_sel] from the selection under test (any device); targets: one
    (b, h_kv, needle key position, t') per query row a needle was aimed at.  A row hits
    when the block of the needle's key, position // C, is among the row's selected blocks.
    Returns {"rows": number of rows, "hit_rate": share of hits, None without rows}."""
    tg = torch.as_tensor([tuple(int(v) for v in x) for x in targets], dtype=torch.int64).reshape(-1, 4)
    if tg.shape[0] == 0:
        return {"rows": 0, "hit_rate": None}
    tg = tg.to(idx.device)
    sel = idx[tg[:, 0], tg[:, 1], tg[:, 3]].to(torch.int64)                 # [R, K_sel]
    hit = (sel == (tg[:, 2] // C)[:, None]).any(dim=1)
    return {"rows": int(tg.shape[0]), "hit_rate": float(hit.double().mean())}
