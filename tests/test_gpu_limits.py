"""Index arithmetic at the top of the supported ranges.

One latent-layout tensor of 2^27 - 1 blocks of 16 slots with 16-byte rows (32 GiB): slots up
to 2^31 - 17 (the largest below the 2^31 limit), block ids near 2^27 and byte offsets past
2^32.  The test writes new tokens into the top slots, builds runs over block ids next to the
top, packs them and unpacks them onto other top blocks.  Each touched row is checked against
the slot formula on the host (slot = block * block_size + offset; block b, slot o at byte
(b * block_size + o) * row_bytes).  The oracle would need the whole 32 GiB on the host, so
these few rows are compared one by one instead.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_kv_cache_81_gb300 import pagedkv as K

pytestmark = pytest.mark.gpu

NB = 2 ** 27 - 1  # blocks: NB * BS = 2^31 - 16 slots
BS = 16
ROW = 16  # bytes per token row: 8 bf16


@pytest.fixture(scope="module")
def big_cache():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_81_gb300 import build
    build.build()
    K.load()
    free, _ = torch.cuda.mem_get_info()
    if free < NB * BS * ROW + (4 << 30):
        pytest.skip("needs 36 GiB of free device memory")
    t = torch.empty((NB, BS, ROW // 2), dtype=torch.bfloat16, device="cuda")
    yield t
    del t
    torch.cuda.empty_cache()


def _rows(t, blocks, offs):
    """uint8 copies of rows (block, offset) of the cache."""
    b = torch.tensor(blocks, dtype=torch.int64, device="cuda")
    o = torch.tensor(offs, dtype=torch.int64, device="cuda")
    return t[b, o].view(torch.uint8).cpu().numpy()


def test_top_slots_written(big_cache):
    t = big_cache
    cache = K.PagedCache.from_tensors([t], "mla")
    assert cache.desc().num_blocks == NB
    # slot_mapping at the top: one request whose table points at the last blocks
    table = torch.tensor([[NB - 1, NB - 2, 2 ** 26, 3]], dtype=torch.int32, device="cuda")
    pos = [63, 48, 15, 0, 40, 33]  # logical blocks 3, 3, 0, 0, 2, 2
    token_req = torch.zeros(len(pos), dtype=torch.int32, device="cuda")
    token_pos = torch.tensor(pos, dtype=torch.int32, device="cuda")
    slot = torch.empty(len(pos), dtype=torch.int64, device="cuda")
    K.kv_get_last_error(clear=True)
    K.kv_slot_mapping(table, token_req, token_pos, BS, slot)
    torch.cuda.synchronize()
    tab = [NB - 1, NB - 2, 2 ** 26, 3]
    want = [tab[p // BS] * BS + p % BS for p in pos]
    assert slot.cpu().tolist() == want
    assert max(want) == (NB - 1) * BS + 15 == 2 ** 31 - 17
    # the rows land where the formula puts them
    new = torch.from_numpy(np.random.default_rng(3).integers(-2 ** 15, 2 ** 15, size=(len(pos), ROW // 2),
                                                             dtype=np.int16)).cuda().view(torch.bfloat16)
    K.kv_reshape_and_cache(cache, [new], slot)
    torch.cuda.synchronize()
    assert K.kv_get_last_error() == 0
    got = _rows(t, [s // BS for s in want], [s % BS for s in want])
    np.testing.assert_array_equal(got, new.view(torch.uint8).cpu().numpy())
    # one slot past the cache is refused and flagged, and nothing is written for it
    bad = torch.tensor([NB * BS], dtype=torch.int64, device="cuda")
    K.kv_reshape_and_cache(cache, [new[:1]], bad)
    torch.cuda.synchronize()
    assert K.kv_get_last_error() & K.KV_DERR_SLOT


def test_top_blocks_packed_and_unpacked(big_cache):
    t = big_cache
    cache = K.PagedCache.from_tensors([t], "mla")
    rng = np.random.default_rng(4)
    src = [NB - 3, NB - 2, NB - 1, 5, 2 ** 26]  # a run of three ending at the last block, then two singles
    dst = [NB - 12, NB - 11, NB - 10, 2 ** 27 - 20, 11]
    fill = torch.from_numpy(rng.integers(-2 ** 15, 2 ** 15, size=(len(src), BS, ROW // 2), dtype=np.int16)).cuda()
    t[torch.tensor(src, device="cuda")] = fill.view(torch.bfloat16)
    off = torch.tensor([0, 3, 5], dtype=torch.int32, device="cuda")
    src_d = torch.tensor(src, dtype=torch.int32, device="cuda")
    dst_d = torch.tensor(dst, dtype=torch.int32, device="cuda")
    K.kv_get_last_error(clear=True)
    x = K.kv_build_xfer_list(off, src_d, dst_d, 0)
    torch.cuda.synchronize()
    runs = x.host()
    # [NB-3 .. NB-1] -> [NB-12 .. NB-10] is one run; 5 and 2^26 are runs of one block each
    assert runs["count"] == 3
    assert runs["src_block"].tolist() == [NB - 3, 5, 2 ** 26] and runs["n_blocks"].tolist() == [3, 1, 1]
    assert runs["dst_block"].tolist() == [NB - 12, 2 ** 27 - 20, 11]
    stage = torch.empty(len(src) * BS * ROW, dtype=torch.uint8, device="cuda")
    K.kv_pack_blocks(cache, x, len(src), stage, 0, ROW)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(stage.cpu().numpy(), fill.view(torch.uint8).cpu().numpy().reshape(-1))
    K.kv_unpack_blocks(cache, stage, x, len(src), BS, ROW, 0)
    torch.cuda.synchronize()
    assert K.kv_get_last_error() == 0
    got = t[torch.tensor(dst, device="cuda")].view(torch.uint8).cpu().numpy()
    np.testing.assert_array_equal(got, fill.view(torch.uint8).cpu().numpy())
