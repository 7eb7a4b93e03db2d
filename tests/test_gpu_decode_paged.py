"""plx_decode_paged: the split-KV decode over a paged cache.  The pages are a
random permutation of the blocks of a contiguous cache (a host-side layout
change, no arithmetic), so the result must equal plx_decode on the contiguous
cache bit for bit, and the fp64 oracle to the decode tolerance."""
import numpy as np
import pytest

import oracle
import plx_inputs

pytestmark = pytest.mark.gpu


def paged_copy(cache, page, rng, spare=3):
    """[B, H, S, d] -> pages [num_blocks, H, page, d] and a block table
    [B, S // page]: every (b, block) gets a distinct random physical block."""
    B, H, S, d = cache.shape
    nb = S // page
    num_blocks = B * nb + spare
    perm = rng.permutation(num_blocks)[: B * nb].reshape(B, nb).astype(np.int32)
    pages = np.zeros((num_blocks, H, page, d), dtype=cache.dtype)
    for b in range(B):
        for j in range(nb):
            pages[perm[b, j]] = cache[b, :, j * page:(j + 1) * page, :]
    return pages, perm


@pytest.mark.parametrize("page,splits", [(32, 1), (64, 3), (128, 0)])
def test_paged_equals_contiguous(page, splits):
    import torch
    import parameterized_local_linear_02_b300 as plx
    S = 512
    dd = plx_inputs.decode(3, 2, 128, S, seed=page + splits, seqlens=np.array([512, 37, 300]))
    t = dd.device_tensors()
    rng = np.random.default_rng(page)
    kb = dd.bits["k_cache"].view(np.int16)
    vb = dd.bits["v_cache"].view(np.int16)
    kp, table = paged_copy(kb, page, rng)
    vp = np.zeros_like(kp)
    for b in range(3):
        for j in range(S // page):
            vp[table[b, j]] = vb[b, :, j * page:(j + 1) * page, :]
    kpt = torch.from_numpy(kp).view(torch.bfloat16).cuda()
    vpt = torch.from_numpy(vp).view(torch.bfloat16).cuda()
    tab = torch.from_numpy(table).cuda()
    o1, l1 = plx.plx_decode_paged(t["q"], t["rho"], kpt, vpt, tab, t["seqlens"], num_splits=splits,
                                  out_dtype=torch.float32)
    o2, l2 = plx.plx_decode(t["q"], t["rho"], t["k_cache"], t["v_cache"], t["seqlens"], num_splits=splits,
                            out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    res = oracle.decode("stream", dd.q, dd.rho, dd.k_cache, dd.v_cache, dd.seqlens, dd.scale)
    exp = np.stack([np.stack([res[(b, h)][0] for h in range(2)]) for b in range(3)])
    err = np.abs(o1.cpu().numpy() - exp).max() / np.sqrt(np.mean(exp ** 2))
    assert err <= 1e-4, f"paged decode vs oracle: {err:.2e}"


def test_paged_invalid_block_id_is_flagged_not_read():
    """A block id outside [0, num_blocks) is replaced by block 0 on the device
    (the copy never leaves the cache) and reported through the status word."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    dd = plx_inputs.decode(1, 2, 64, 64, seed=5, seqlens=np.array([64]))
    t = dd.device_tensors()
    pages = t["k_cache"].reshape(1, 2, 2, 32, 64).permute(0, 2, 1, 3, 4).reshape(2, 2, 32, 64).contiguous()
    vpages = t["v_cache"].reshape(1, 2, 2, 32, 64).permute(0, 2, 1, 3, 4).reshape(2, 2, 32, 64).contiguous()
    table = torch.tensor([[0, 7]], dtype=torch.int32, device="cuda")     # 7 >= num_blocks = 2
    plx.plx_decode_paged(t["q"], t["rho"], pages, vpages, table, t["seqlens"], num_splits=1)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 1      # PLX_ERR_INVALID_ARG
    assert plx.plx_last_device_error() == 0      # the status word was cleared by the read
