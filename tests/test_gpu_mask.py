"""GPU parity of block_causal_mask against the oracle: additive fp32 / bf16
(0 or -inf, bit-exact) and the 0/1 keep mask, over ragged widths, padded and
unaligned row strides, query / key offsets (windows that do not start at
position 0) and rows wide enough to span several of the kernel's chunks."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def expect(Lq, Lk, bl, qo, ko):
    return oracle.block_causal_mask(Lq, bl, Lk=Lk, q_offset=qo, k_offset=ko)


@pytest.mark.parametrize("Lq,Lk,bl,qo,ko", [(1, 1, 1, 0, 0), (4, 4, 2, 0, 0), (33, 33, 32, 0, 0),
                                            (160, 160, 32, 0, 0), (32, 1024, 32, 992, 0), (100, 257, 7, 3, 5),
                                            (1000, 1000, 1, 0, 0), (64, 64, 4096, 0, 0)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.uint8, torch.bool])
def test_mask_matches_oracle(cs, Lq, Lk, bl, qo, ko, dtype):
    want = expect(Lq, Lk, bl, qo, ko)
    got = cs.block_causal_mask(Lq, bl, Lk=Lk, q_offset=qo, k_offset=ko, dtype=dtype).cpu()
    if dtype in (torch.uint8, torch.bool):
        assert np.array_equal(got.numpy().astype(bool), want == 0)
    else:
        g = got.float().numpy()
        assert np.array_equal(g, want.astype(np.float32))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.uint8])
def test_mask_padded_and_unaligned_rows(cs, dtype):
    Lq, Lk, bl = 70, 130, 16
    want = expect(Lq, Lk, bl, 0, 0)
    for pad, shift in ((6, 0), (0, 1), (3, 3)):
        sentinel = 7
        big = torch.full((Lq, Lk + pad + shift), sentinel, dtype=dtype, device="cuda")
        view = big[:, shift:shift + Lk]
        cs.block_causal_mask(Lq, bl, Lk=Lk, dtype=dtype, out=view)
        g = view.cpu().float().numpy()
        if dtype == torch.uint8:
            assert np.array_equal(g.astype(bool), want == 0)
        else:
            assert np.array_equal(g, want.astype(np.float32))
        rest = torch.cat([big[:, :shift], big[:, shift + Lk:]], dim=1).cpu().float().numpy()
        assert np.all(rest == sentinel)


def test_mask_rejects_bad_arguments(cs):
    out = torch.empty((4, 4), device="cuda")
    with pytest.raises(cs.DllmError):
        cs.block_causal_mask(4, 0, out=out)
    with pytest.raises(cs.DllmError):
        cs.block_causal_mask(4, 2, q_offset=-1, out=out)


# rows of several 16 KiB chunks: 40009 columns are 10002 fp32 vectors (ten
# chunks of 1024, the last partial, one element past them), 5001 bf16 vectors
# and 2500 keep-mask vectors (three chunks), each with a ragged tail
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.uint8])
def test_mask_rows_of_several_chunks(cs, dtype):
    Lq, Lk, bl, qo, ko = 5, 40009, 3, 30000, 1001   # the attend runs end inside a vector
    want = expect(Lq, Lk, bl, qo, ko)
    got = cs.block_causal_mask(Lq, bl, Lk=Lk, q_offset=qo, k_offset=ko, dtype=dtype).cpu()
    if dtype == torch.uint8:
        assert np.array_equal(got.numpy().astype(bool), want == 0)
    else:
        assert np.array_equal(got.float().numpy(), want.astype(np.float32))
    # padded and unaligned strides on the same widths leave the rest untouched
    for pad, shift in ((16, 0), (0, 1)):
        sentinel = 7
        big = torch.full((Lq, Lk + pad + shift), sentinel, dtype=dtype, device="cuda")
        view = big[:, shift:shift + Lk]
        cs.block_causal_mask(Lq, bl, Lk=Lk, q_offset=qo, k_offset=ko, dtype=dtype, out=view)
        g = view.cpu().float().numpy()
        if dtype == torch.uint8:
            assert np.array_equal(g.astype(bool), want == 0)
        else:
            assert np.array_equal(g, want.astype(np.float32))
        rest = torch.cat([big[:, :shift], big[:, shift + Lk:]], dim=1).cpu().float().numpy()
        assert np.all(rest == sentinel)
