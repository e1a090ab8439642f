"""Token samples for the full-size parity checks, and the oracle on them.

At the full workload sizes the oracle cannot recompute every token, but each
token's output depends only on its own hidden row and its k experts, so the
oracle runs on a sample.  The sample is chosen to reach every tile the
grouped GEMMs cut the expert-sorted rows into:

* for the expert with the most rows, the first and the last row of every
  128-row tile of the token-row GEMM, of every near-equal token tile of the
  swap-AB GEMM (at most 128 rows) and of every near-equal token tile of the
  CTA-pair GEMM (at most 256 rows), so both sides of every tile boundary,
  and the last tile;
* for every other touched expert, its first and last row.

A row stands for its token.  With ``cheap`` (a set of experts), only tokens
whose k experts all lie in that set are used, taking the eligible row
nearest each tile edge; this bounds how many experts the oracle has to
dequantise.

The check itself is made on the fp32 accumulator the grouped paths sum
into (read back from the workspace): it must be within the tolerance of the
oracle, and the bf16 output must be exactly its round-to-nearest-even image.
Comparing the bf16 output with the oracle directly would also charge the
output's own rounding to the kernels: at millions of outputs the largest
reach several times rms, where half a bf16 unit (up to 2^-8 of the value)
alone approaches 2e-2 of rms.

Test infrastructure: uses the oracle and the library's binding, never the
library's arithmetic.
"""
import numpy as np
import torch

import oracle as O

TILE_ROWS = 128
PAIR_TILE_ROWS = 256


def _segments(o, M):
    """Row ranges of the tiles of one expert (rows [o, o+M))."""
    segs = [(o + b, o + min(b + TILE_ROWS, M)) for b in range(0, M, TILE_ROWS)]
    for rows in (TILE_ROWS, PAIR_TILE_ROWS):
        ntt = -(-M // rows)
        segs += [(o + j * M // ntt, o + (j + 1) * M // ntt) for j in range(ntt)]
    return segs


def tile_count(M):
    """Number of tile row ranges of an expert with M rows (see _segments)."""
    return 2 * -(-M // TILE_ROWS) + -(-M // PAIR_TILE_ROWS)


def probe_tokens(ref_idx, E, k, cheap=None):
    """Sorted token indices of the tile-edge sample (see the module text).
    Returns (tokens, counts, hot expert, number of tiles of the hot expert
    reached by the sample)."""
    counts, offsets, sorted_f, _ = O.dispatch(ref_idx, E)
    tok_of_row = sorted_f.astype(np.int64) // k
    if cheap is None:
        ok_tok = np.ones(ref_idx.shape[0], bool)
    else:
        cheap_mask = np.zeros(E, bool)
        cheap_mask[list(cheap)] = True
        ok_tok = cheap_mask[ref_idx].all(axis=1)
    ok_row = ok_tok[tok_of_row]
    hot = int(np.argmax(counts))
    toks = set()
    reached = 0
    for e in range(E):
        M = int(counts[e])
        if M == 0 or (cheap is not None and e not in cheap):
            continue
        o = int(offsets[e])
        segs = _segments(o, M) if e == hot else [(o, o + M)]
        for a, b in segs:
            rows = np.nonzero(ok_row[a:b])[0]
            if rows.size:
                toks.add(int(tok_of_row[a + rows[0]]))
                toks.add(int(tok_of_row[a + rows[-1]]))
                reached += e == hot
    return np.array(sorted(toks), np.int64), counts, hot, reached


def oracle_on_tokens(toks, ref_idx, ref_w, hidden_rows, expert_fn):
    """out[i] = sum_j ref_w[t, j] * y_j for the sampled tokens t = toks[i],
    where expert_fn(e, x) returns the expert's output rows y for input rows
    x (float64 [n, H])."""
    sub = ref_idx[toks]
    wsub = np.asarray(ref_w, np.float64)[toks]
    out = np.zeros((len(toks), hidden_rows.shape[1]), np.float64)
    for e in np.unique(sub):
        rt, rj = np.nonzero(sub == e)          # a token lists an expert at most once
        y = expert_fn(int(e), hidden_rows[rt])
        out[rt] += wsub[rt, rj][:, None] * y
    return out


def bf16_expert_fn(w_gate_up, w_down):
    """Expert MLP through the oracle's forward on one expert (k = 1, weight 1,
    float32 as for every full-size check), weights copied per expert."""
    def fn(e, x):
        wgu = w_gate_up[e].float().cpu().numpy()[None]
        wd = w_down[e].float().cpu().numpy()[None]
        n = x.shape[0]
        return O.forward(x, np.zeros((n, 1), np.int32), np.ones((n, 1)), wgu, wd,
                         dtype=np.float32)
    return fn


def fp8_expert_fn(q_gate_up, s_gate_up, q_down, s_down, fmt):
    """The mirrored FP8 forward on one expert (same block-scaled weights,
    same dynamic activation and h quantisation)."""
    def fn(e, x):
        n = x.shape[0]
        sl = slice(e, e + 1)
        return O.forward_fp8(x.astype(np.float32), np.zeros((n, 1), np.int32), np.ones((n, 1)),
                             q_gate_up[sl].cpu().numpy(), s_gate_up[sl].cpu().numpy(),
                             q_down[sl].cpu().numpy(), s_down[sl].cpu().numpy(), fmt)
    return fn


def check_accumulator(moe, out, toks, ref, shape, wdtype, tol, workspace=None):
    """The fp32 accumulator rows of the sampled tokens are within ``tol``
    (max |err| / rms) of the oracle, and out holds their bf16 RNE images.
    Returns (accumulator error, bf16 output error against the rounded
    oracle) for the message of a failing assertion."""
    ws = moe.default_workspace() if workspace is None else workspace
    acc = moe.accumulator(ws, shape.T, shape.H, shape.I, shape.E, shape.k, wdtype)
    tt = torch.from_numpy(np.asarray(toks)).to(out.device)
    acc_s = acc[tt].cpu().numpy()
    got = out[tt].float().cpu().numpy()
    err_acc = O.rel_max_err(acc_s, ref)
    err_out = O.rel_max_err(got, O.round_to_bf16(ref))
    assert np.array_equal(got, O.round_to_bf16(acc_s)), "bf16 output is not the RNE image of the accumulator"
    assert err_acc <= tol, (err_acc, err_out)
    return err_acc, err_out
