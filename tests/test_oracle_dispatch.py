"""Pins of the oracle's local expert dispatch (routing of top-k choices to
expert groups, MXFP4 quantization of the routed rows, padded or slot scale
layout) -- "Struct_ep_dispatch_mxfp4", execute -- against hand-worked cases,
a library stable sort and layout identities."""
import numpy as np

from oracle import dispatch as D
from oracle import layout as L
from oracle import quantize as Q


def test_route_hand_case():
    # token 0 -> experts (2, 0), token 1 -> (1, 2), token 2 -> (0, 0)
    # choices i = 0..5 go to experts 2, 0, 1, 2, 0, 0
    ro, eids, src, dropped = D.route_topk([[2, 0], [1, 2], [0, 0]], 3)
    assert ro.tolist() == [0, 3, 4, 6]
    assert eids.tolist() == [0, 1, 2]
    assert src.tolist() == [1, 4, 5, 2, 0, 3]
    assert dropped == 0


def test_route_drops_invalid_ids_and_keeps_empty_groups():
    # experts 0..3; ids -1 and 4 are dropped; expert 1 receives nothing
    ro, eids, src, dropped = D.route_topk([[3, -1], [4, 0], [3, 2]], 4)
    assert ro.tolist() == [0, 1, 1, 2, 4]
    assert src.tolist() == [3, 5, 0, 4]
    assert dropped == 2
    assert eids.tolist() == [0, 1, 2, 3]


def test_route_matches_a_stable_sort():
    rng = np.random.default_rng(7)
    for E, T, k in [(8, 129, 2), (256, 64, 8), (5, 1000, 3)]:
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        ro, _, src, dropped = D.route_topk(ids, E)
        flat = ids.reshape(-1)
        assert dropped == 0
        assert np.array_equal(src, np.argsort(flat, kind="stable"))
        assert np.array_equal(np.diff(ro.astype(np.int64)), np.bincount(flat, minlength=E))


def test_slot_offsets():
    assert D.slot_scale_offsets(3, 256).tolist() == [0, 256, 512, 768]


def _tokens(T, H, seed):
    rng = np.random.default_rng(seed)
    # bf16-representable values, distinct rows
    x = rng.normal(size=(T, H)).astype(np.float32)
    return (x.view(np.uint32) & 0xFFFF0000).view(np.float32) * (1 + np.arange(T))[:, None]


def test_dispatch_routes_tokens_not_choices():
    # top_k = 2: routed row r must be token src[r] // 2
    tok = _tokens(3, 64, 1)
    out = D.dispatch_mxfp4(tok, [[1, 0], [0, 1], [1, 0]], 2)
    src = out["src_info"]
    assert src.tolist() == [1, 2, 5, 0, 3, 4]
    q_ref, _ = Q.quantize_rows("mxfp4", tok[src // 2])
    assert np.array_equal(out["q"], q_ref)
    # rows of distinct tokens differ, so a wrong divisor would show
    assert not np.array_equal(q_ref[0], q_ref[1])


def test_slot_layout_holds_the_same_scales_as_the_padded_layout():
    tok = _tokens(40, 128, 2)
    rng = np.random.default_rng(3)
    ids = np.stack([rng.choice(4, 2, replace=False) for _ in range(40)]).astype(np.int32)
    a = D.dispatch_mxfp4(tok, ids, 4)
    b = D.dispatch_mxfp4(tok, ids, 4, max_padded_m=128)
    assert np.array_equal(a["q"], b["q"])
    ro = a["row_offsets"]
    kv = 128 // 32
    for g in range(4):
        for r in range(int(ro[g]), int(ro[g + 1])):
            for c in range(kv):
                pa = L.sf_offset(int(a["scales_offsets"][g]) + r - int(ro[g]), c, kv)
                pb = L.sf_offset(int(b["scales_offsets"][g]) + r - int(ro[g]), c, kv)
                assert a["scales"][pa] == b["scales"][pb]
    assert b["scales"].size == L.physical_bytes(4 * 128, kv)


def test_topk_amax_hand_case():
    # token amaxes 3, 2, 4; expert 0 <- tokens 0, 2; 1 <- 0, 1; 2 <- 1, 2; 3 <- none
    tok = np.array([[1, -3], [2, 0.5], [-4, 1]], np.float32)
    amax = D.topk_amax(tok, [[0, 1], [1, 2], [2, 0]], 4)
    assert amax.tolist() == [4.0, 3.0, 4.0, 0.0]
    # an id outside the experts is dropped
    assert D.topk_amax(tok, [[0, 9], [1, -1], [1, 0]], 2).tolist() == [4.0, 4.0]


def test_topk_amax_equals_the_grouped_amax_of_the_routed_rows():
    rng = np.random.default_rng(11)
    tok = _tokens(50, 64, 12)
    ids = np.stack([rng.choice(9, 3, replace=False) for _ in range(50)]).astype(np.int32)
    ro, eids, src, _ = D.route_topk(ids, 9)
    ref = Q.group_amax(tok[src // 3], ro, eids, 9)
    assert np.array_equal(D.topk_amax(tok, ids, 9), ref)
