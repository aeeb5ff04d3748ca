"""The CPU oracle over many independent pieces of work at once (test helper).

Tokens are independent, and so are the layers of a chain once the GPU's input
to each layer is known, so a large parity check splits into pieces that run
in separate processes, each calling the single-threaded oracle as it stands.
The pool uses the ``spawn`` start method: a process forked after CUDA has been
initialised in the parent would hang.

Each piece is (workload name, layer, x bits [T][H], ids [T][k] or None, router
rows, shared-gate vector, logit offsets or None). A worker routes x with the
oracle (keeping the probabilities) and combines the experts named by ``ids``
(the GPU's choice) with the weights the method gives that choice: the oracle's
probabilities of those experts, renormalised over them. With ids=None it
combines the oracle's own choice. 8-bit workloads use the oracle's 8-bit
combine.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np


def own_choice_weights(probs: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """w[t][j] = p[t][ids[t][j]] / sum_i p[t][ids[t][i]] (fp64): the top-k
    renormalisation applied to a given choice of experts."""
    sel = np.take_along_axis(probs, ids.astype(np.int64), axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


def layer_piece(args):
    """One piece of work (see the module docstring). Returns a dict with the
    oracle's ids, w, gate, probs, and out64 of the combined choice and the
    weights used for it (w_used)."""
    import synthetic
    import oracle
    name, layer, x, ids, Wr, ws, bias = args
    wl = synthetic.WORKLOADS[name]
    r_ids, r_w, r_gate, probs = oracle.route(x, Wr, ws, wl.k, bias=bias, want_probs=True)
    use = r_ids if ids is None else np.ascontiguousarray(ids, np.int32)
    w_used = r_w if ids is None else own_choice_weights(probs, use)
    bits = wl.bits
    experts = {int(e): synthetic.expert_triples(wl.seed, layer, int(e), wl.H, wl.I, bits=bits) for e in np.unique(use)}
    shared = synthetic.expert_triples(wl.seed, layer, None, wl.H, wl.I_shared, bits=bits)
    combine = oracle.combine8 if bits == 8 else oracle.combine
    out64, outb = combine(x, use, w_used, r_gate, experts, shared, wl.E, wl.I, wl.I_shared)
    return dict(ids=r_ids, w=r_w, gate=r_gate, probs=probs, out64=out64, out_bf16=outb, w_used=w_used)


def workers() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def run_pieces(pieces):
    """layer_piece over every piece, in parallel processes; results in order."""
    if len(pieces) == 1:
        return [layer_piece(pieces[0])]
    with ProcessPoolExecutor(max_workers=min(workers(), len(pieces)), mp_context=mp.get_context("spawn")) as ex:
        return list(ex.map(layer_piece, pieces))


def tokens_sharded(name, layer, x, ids, Wr, ws, bias=None, shards=None):
    """layer_piece over the tokens of x split into contiguous shards, merged
    back in token order."""
    T = x.shape[0]
    n = min(T, shards or workers())
    cuts = np.linspace(0, T, n + 1).astype(int)
    pieces = [(name, layer, np.ascontiguousarray(x[a:b]), None if ids is None else np.ascontiguousarray(ids[a:b]),
               Wr, ws, bias) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
    parts = run_pieces(pieces)
    return {key: np.concatenate([p[key] for p in parts], axis=0) for key in parts[0]}
