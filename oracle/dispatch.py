"""Local part of the expert-parallel MXFP4 token dispatch
("Struct_ep_dispatch_mxfp4", execute).

TEST INFRASTRUCTURE ONLY (see the package docstring).

With a single rank the all-to-all exchange of the dispatch is the identity;
what remains is (1) routing every (token, slot) choice of ``topk_ids`` to the
group of its expert -- the row offsets, expert ids and source information the
page lists among the outputs -- and (2) quantizing the routed rows to MXFP4,
the activation scales written either in the padded per-expert layout of the
grouped quantizer or, with the scale-slot fusion (fuse_a_scale_preshuffle),
into fixed-stride per-expert slots of max_padded_M rows.

Readings (the page names the outputs, not their order or content):

* group e is expert e for every e in [0, E), empty groups included:
  expert_ids = 0..E-1 and row_offsets has E + 1 entries;
* a group's rows hold its choices in increasing choice index
  i = t * top_k + k (a stable order; the page's atomic counters leave the
  order open);
* src_info[r] = i, the choice held by row r (token i // top_k, slot
  i % top_k); the routed row is token i // top_k;
* a choice whose expert id lies outside [0, E) is dropped;
* slot layout: group g's scale rows start at g * max_padded_M.
"""
import numpy as np

from . import quantize as Q


def route_topk(topk_ids, num_experts):
    """Returns (row_offsets uint32 [E+1], expert_ids int32 [E],
    src_info int32 [routed choices], dropped choices)."""
    ids = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    E = int(num_experts)
    rows_of = [[] for _ in range(E)]
    dropped = 0
    for i, e in enumerate(ids.tolist()):   # choices in increasing i
        if 0 <= e < E:
            rows_of[e].append(i)
        else:
            dropped += 1
    counts = [len(r) for r in rows_of]
    row_offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.uint32)
    src_info = np.array([i for r in rows_of for i in r], dtype=np.int32)
    return row_offsets, np.arange(E, dtype=np.int32), src_info, dropped


def topk_amax(tokens, topk_ids, num_experts):
    """Per-expert amax from tokens and their top-k choices: amax_e = max |x_t|
    over the tokens t with a choice of expert e (0 when there is none); ids
    outside [0, E) are dropped.  The same set of values as the grouped amax
    over the routed rows ("grouped_quantize_dynamic_scaled_fp4_async_kernel":
    the per-expert tensor scale comes from the expert's rows)."""
    x = np.asarray(tokens, dtype=np.float32)
    ids = np.asarray(topk_ids, dtype=np.int64)
    if ids.ndim != 2:
        ids = ids.reshape(x.shape[0], -1)
    amax = np.zeros(int(num_experts), dtype=np.float32)
    for t in range(x.shape[0]):
        m = np.abs(x[t]).max() if x.shape[1] else np.float32(0)
        for e in ids[t]:
            if 0 <= e < num_experts:
                amax[e] = max(amax[e], m)
    return amax


def slot_scale_offsets(num_experts, max_padded_m):
    """scales_offsets of the slot layout: group g starts at g * max_padded_M."""
    return (np.arange(int(num_experts) + 1, dtype=np.int64) * int(max_padded_m)).astype(np.uint32)


def dispatch_mxfp4(tokens, topk_ids, num_experts, max_padded_m=0, scale_rows_total=None):
    """The dispatch on one rank.  tokens: [num_tokens, hidden] float32 holding
    BF16 values; topk_ids: [num_tokens, top_k].  Returns a dict with the
    routing, the scale offsets used, the packed MXFP4 rows
    [num_tokens * top_k, hidden / 2] (rows of dropped choices zero) and the
    tiled E8M0 scale buffer of scale_rows_total logical rows."""
    tokens = np.asarray(tokens, dtype=np.float32)
    top_k = np.asarray(topk_ids).reshape(tokens.shape[0], -1).shape[1]
    ro, eids, src, dropped = route_topk(topk_ids, num_experts)
    if max_padded_m:
        so = slot_scale_offsets(num_experts, max_padded_m)
    else:
        so = Q.padded_scale_offsets(ro)
    if scale_rows_total is None:
        scale_rows_total = int(so[-1])
    T = tokens.shape[0] * top_k
    x = np.zeros((T, tokens.shape[1]), np.float32)
    x[:len(src)] = Q.gather_rows(tokens, src, top_k)
    q, sc = Q.grouped_quantize("mxfp4", x, ro, so, eids, scale_rows_total=scale_rows_total)
    q[len(src):] = 0
    return {"row_offsets": ro, "expert_ids": eids, "src_info": src, "dropped": dropped,
            "scales_offsets": so, "q": q, "scales": sc}
