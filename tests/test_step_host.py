"""Host-side arithmetic of the step that needs no GPU.

TransferStep sizes the staging buffer of a sliding-window step from the host's copy of the
request lengths (TransferStep.kept_blocks), without reading the clip kernel's count back.  If
that count drifted from the clip rule, the staging buffer and the listed-block count would be
wrong silently, so it is compared here with the oracle's clip (Mooncake page, section 3.1,
get_sw_clipped_blocks; the reading: entries max(0, n - window) / bs .. ceil(n / bs) - 1, never
past the list, window <= 0 keeps every entry holding a token) over random inputs.
"""
from __future__ import annotations

import numpy as np

import oracle
from paged_kv_cache_81_gb300 import workloads as W
from paged_kv_cache_81_gb300.step import TransferStep


def test_kept_blocks_equals_the_oracle_clip_count():
    rng = np.random.default_rng(8181)
    for trial in range(400):
        bs = int(rng.choice([1, 2, 3, 16, 64]))
        R = int(rng.integers(0, 12))
        lens = rng.integers(0, 40, size=R)
        lists = W.pop_lists(rng.permutation(int(lens.sum()) + 1), lens) if R else []
        # token counts from empty to past the list's capacity (the clip never runs past the list)
        n_tok = np.array([int(rng.integers(0, l * bs + 2 * bs + 1)) for l in lens], dtype=np.int32)
        window = int(rng.choice([-3, 0, 1, bs - 1, bs, bs + 1, 5 * bs, 37, 10 ** 6]))
        off, ids = W.csr(lists)
        case = W.Case(W.TINY, off, ids, off, ids, req_tokens=n_tok)
        out_off, kept_ids = oracle.clip_block_lists(off, ids, n_tok, window, bs)
        want = int(out_off[-1])
        assert kept_ids.shape[0] == want
        got = TransferStep.kept_blocks(case, window, bs)
        assert got == want, (trial, bs, window, lens.tolist(), n_tok.tolist())
