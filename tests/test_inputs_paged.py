"""The paged layout the input generator draws (host only): every block that
holds rows of a sequence maps to a distinct page, blocks past a sequence are
unmapped (-1), pages no table names stay NaN, and each mapped page holds the
rows of its block."""
import torch

from compressed_cache_decode_gb300 import inputs


def test_paged_layout_invariants():
    case = inputs.random_decode_case(seed=3, batch=3, heads=2, head_dim=16, rank=4, max_len=64, dtype="bf16",
                                     lens=[64, 17, 0])
    ps = 16
    paged = inputs.paged_from_contiguous(case, page_size=ps, seed=5, extra_pages=2)
    bt = paged["block_table"]
    assert bt.dtype == torch.int32 and tuple(bt.shape) == (3, 4)
    lens = case["seq_lens"].tolist()
    mapped = []
    for b in range(3):
        for j in range(4):
            if j * ps < lens[b]:
                assert bt[b, j] >= 0
                mapped.append(int(bt[b, j]))
                for name in ("k_s", "z_v"):
                    assert torch.equal(paged[name][bt[b, j]].view(torch.int16),
                                       case[name][b, j * ps:(j + 1) * ps].view(torch.int16))
            else:
                assert bt[b, j] == -1
    assert len(set(mapped)) == len(mapped) == 4 + 2 + 0
    pool_pages = paged["k_s"].shape[0]
    assert pool_pages == len(mapped) + 2
    for pg in set(range(pool_pages)) - set(mapped):
        assert torch.isnan(paged["k_s"][pg].float()).all()
