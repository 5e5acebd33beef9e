"""Host-side block-mask builder (fa_block_mask_build): classes and bitmasks
reproduce the dense mask exactly.  CPU only."""
import numpy as np
import pytest

from flash_attention_gqa_gb300 import binding
import os


@pytest.fixture(scope="module")
def clib():
    if not os.path.exists(binding.LIB_PATH):
        from flash_attention_gqa_gb300 import build
        build.build()
    return binding.load()


def expand(cls, idx, bits, T, S):
    heads, nqb, nkb = cls.shape
    out = np.zeros((heads, nqb * 128, nkb * 128), dtype=bool)
    bits = bits.numpy().view(np.uint32) if hasattr(bits, "numpy") else bits
    for h in range(heads):
        for qb in range(nqb):
            for kb in range(nkb):
                c = int(cls[h, qb, kb])
                blk = out[h, qb * 128:(qb + 1) * 128, kb * 128:(kb + 1) * 128]
                if c == 1:
                    blk[:] = True
                elif c == 2:
                    w = bits[int(idx[h, qb, kb])]                       # [128, 4]
                    for j in range(128):
                        blk[:, j] = (w[:, j // 32] >> (j % 32)) & 1
    return out[:, :T, :S]


@pytest.mark.parametrize("T,S", [(128, 128), (300, 260), (5, 700)])
def test_builder_round_trip(clib, T, S):
    rng = np.random.default_rng(T + S)
    heads = 3
    dense = rng.random((heads, T, S)) < 0.5
    dense[0, :128, :] = False                       # whole empty blocks
    dense[1, :, :128] = True                        # whole full blocks
    cls, idx, bits, h = binding.block_mask_from_dense(dense)
    cls, idx = cls.numpy(), idx.numpy()
    assert h == heads
    assert np.array_equal(expand(cls, idx, bits, T, S), dense)
    assert np.all(cls[0, 0, :] == 0) and np.all(cls[1, :, 0] == 1)
    assert np.all((idx >= 0) == (cls == 2))


def test_builder_rejects_small_capacity(clib):
    dense = np.zeros((1, 128, 128), dtype=np.uint8)
    dense[0, 0, 0] = 1
    cls = np.zeros((1, 1, 1), np.uint8)
    idx = np.zeros((1, 1, 1), np.int32)
    rc, n = binding.fa_block_mask_build(dense, 1, 128, 128, cls, idx, None, 0)
    assert rc == binding.FA_OK and n == 1
    bits = np.zeros((1, 128, 4), np.uint32)
    rc, n = binding.fa_block_mask_build(dense, 1, 128, 128, cls, idx, bits, 0)
    assert rc == binding.FA_ERR_INVALID_ARG
