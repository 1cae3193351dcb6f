"""Pins for the oracle's expert-parallel dispatch metadata (the receiving side's expert of each
received row).

Independent reference: the single-process layer. Expert parallelism over G simulated ranks --
route and permute on each source, the rows of each destination's experts sent to it, the
receiving side's expert ids and a local permute, each local expert's MLP, the rows sent back
and combined at the source -- must give every rank exactly the output the oracle's
single-process layer gives for its tokens (every row meets the same expert with the same
operands). Experts have distinct weights, so a row sent to the wrong expert shows."""
import numpy as np
import pytest
import torch

import oracle as O


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _mlp(x_bits, w, off, E):
    """The oracle's grouped SwiGLU MLP on every row of x_bits (bf16 h) -> y bf16 bits."""
    w1, w3, w2 = w
    R = int(off[-1])
    out = np.zeros((x_bits.shape[0], w1.shape[1]), np.uint16)
    if R:
        rows = np.arange(R, dtype=np.int32)
        y = O.swiglu_rows(O.Operand(O.MAT_BF16, x_bits), O.Operand(O.MAT_BF16, w1), O.Operand(O.MAT_BF16, w3),
                          O.Operand(O.MAT_BF16, w2), off, rows, h_mode=O.H_BF16, want=("y_bf16",))["y_bf16"]
        out[:R] = y
    return out


def _single(x, lg, w, E, K, renorm):
    ids, probs = O.route_topk(lg, K, renorm)
    op = O.permute(x, ids, E)
    y_perm = _mlp(op["x_perm"], w, op["group_offsets"], E)
    return O.combine(y_perm, op["row_map"], probs)


def _ep(xs, lgs, w, E, K, G, renorm):
    E_loc = E // G
    src = []
    for x, lg in zip(xs, lgs):
        ids, probs = O.route_topk(lg, K, renorm)
        op = O.permute(x, ids, E)
        src.append((ids, probs, op))
    # dispatch: destination g receives, source by source, the rows of experts g*E_loc..
    recv = []
    for g in range(G):
        counts = np.stack([op["group_sizes"][g * E_loc:(g + 1) * E_loc] for _, _, op in src])
        rows = np.concatenate([op["x_perm"][op["group_offsets"][g * E_loc]:op["group_offsets"][(g + 1) * E_loc]]
                               for _, _, op in src])
        N = rows.shape[0]
        lid = O.ep_recv_expert_ids(counts, N + 3)              # three rows of spare capacity
        assert np.all(lid[N:] == -1)
        rows_cap = np.concatenate([rows, np.zeros((3, rows.shape[1]), np.uint16)])
        loc = O.permute(rows_cap, lid[:, None], E_loc)          # local expert order, K = 1
        assert np.array_equal(loc["group_sizes"], counts.sum(axis=0))
        wl = tuple(t[g * E_loc:(g + 1) * E_loc] for t in w)
        y_loc = _mlp(loc["x_perm"], wl, loc["group_offsets"], E_loc)
        y_recv = O.permute_backward(y_loc, loc["row_map"])     # back to the received order
        recv.append((counts, y_recv))
    # combine: each source takes its rows back, in its own permuted order
    outs = []
    for s, (ids, probs, op) in enumerate(src):
        parts = []
        for g in range(G):
            counts, y_recv = recv[g]
            start = int(counts[:s].sum())
            parts.append(y_recv[start:start + int(counts[s].sum())])
        y_back = np.concatenate(parts + [np.zeros((ids.size - op["R"], parts[0].shape[1]), np.uint16)])
        outs.append(O.combine(y_back, op["row_map"], probs))
    return outs


@pytest.mark.parametrize("G,E,K,renorm", [(2, 6, 2, True), (3, 6, 3, False), (1, 4, 2, False), (4, 8, 1, True)])
def test_ep_over_simulated_ranks_equals_single_process_layer(G, E, K, renorm):
    rng = np.random.default_rng(G * 10 + E)
    H = F = 32
    T = 40
    w = tuple(_bf16(rng.standard_normal(s) * 0.3) for s in ((E, H, F), (E, H, F), (E, F, H)))
    xs = [_bf16(rng.standard_normal((T, H))) for _ in range(G)]
    lgs = [(rng.standard_normal((T, E)) + rng.standard_normal(E)).astype(np.float32) for _ in range(G)]
    lgs[0][:5] = lgs[0][0]            # equal rows: identical routes from several tokens
    got = _ep(xs, lgs, w, E, K, G, renorm)
    for x, lg, y in zip(xs, lgs, got):
        assert np.array_equal(y, _single(x, lg, w, E, K, renorm))


def test_recv_expert_ids_segments_and_capacity():
    counts = np.array([[2, 0, 1], [0, 3, 1]], np.int32)
    assert O.ep_recv_expert_ids(counts, 9).tolist() == [0, 0, 2, 1, 1, 1, 2, -1, -1]
    assert O.ep_recv_expert_ids(counts, 4).tolist() == [0, 0, 2, 1]        # capacity cuts the tail
    assert O.ep_recv_expert_ids(np.zeros((3, 2), np.int32), 2).tolist() == [-1, -1]
