"""The full-size parity tests recompute chosen tokens with the oracle as
smaller oracle transfers (``parity.oracle_tokens``).  Here, on the CPU, those
token-subset results must equal the full oracle transfer's rows bit for bit,
for a ragged paged batch with per-request offsets and for the wide map."""
import dataclasses

import numpy as np

import oracle
from cross_model_kv_transfer_gb300.workloads import WORKLOADS, make_inputs, make_wide_weights

from parity import dst_rows_of, oracle_tokens, run_oracle


def _small_paged():
    return dataclasses.replace(
        WORKLOADS["llama31_8b_70b_paged"].with_tokens([37, 5, 70], [3, 64, 0]),
        src_layers=5, tgt_layers=3, kv_heads=2, head_dim=16, k=2)


def test_token_subsets_equal_the_full_transfer_rows():
    wl = _small_paged()
    inp = make_inputs(wl, "cpu")
    full_k, full_v, st = run_oracle(wl, inp)
    assert st == 0
    tokens = [0, 1, 2, 36, 37, 40, 41, 42, 43, 50, 111, 80]   # runs across request edges
    ok, ov, toks = oracle_tokens(wl, inp, tokens, threads=3)
    assert list(toks) == sorted(set(tokens))
    rows = dst_rows_of(wl, inp, toks)
    assert np.array_equal(ok, full_k[:, rows]) and np.array_equal(ov, full_v[:, rows])
    # every token of the batch, one thread per token
    all_tok = np.arange(wl.ntok)
    ok, ov, _ = oracle_tokens(wl, inp, all_tok, threads=8)
    rows = dst_rows_of(wl, inp, all_tok)
    written = ~np.isnan(full_k[..., 0, 0])
    assert written.sum(axis=1).tolist() == [wl.ntok] * wl.tgt_layers
    assert np.array_equal(ok, full_k[:, rows]) and np.array_equal(ov, full_v[:, rows])


def test_token_subsets_of_the_wide_map_equal_the_full_transfer_rows():
    wl = dataclasses.replace(_small_paged(), layout=0)
    wl = dataclasses.replace(wl, tgt_offsets=(0, 4, 9))
    inp = make_inputs(wl, "cpu")
    inp["w"] = make_wide_weights(wl, "cpu")
    full_k, full_v, st = run_oracle(wl, inp, wide=True)
    assert st == 0
    tokens = [3, 4, 5, 41, 100, 111]
    ok, ov, toks = oracle_tokens(wl, inp, tokens, threads=2, wide=True)
    rows = dst_rows_of(wl, inp, toks)
    assert np.array_equal(ok, full_k[:, rows]) and np.array_equal(ov, full_v[:, rows])
