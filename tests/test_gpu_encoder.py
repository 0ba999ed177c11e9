"""GPU trellis encoder against the CPU oracle: the words are bit-identical
(every Viterbi decision is integer) and so are the per-tile errors; the
decoded weights of the GPU's words, through the layer's own debug decode, give
back the reported error."""
import numpy as np
import pytest
import torch

import exl3_trellis_quantized_rot_gb300 as tfx
import oracle
from gpu_helpers import DEV

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build_library()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def grid_targets(seed, K, N, sigma=1.155):
    rng = np.random.default_rng(seed)
    return np.clip(np.rint(rng.normal(0.0, sigma, (K, N)) * 128), -1024, 1023).astype(np.int16)


@pytest.mark.parametrize("bits", range(1, 9))
def test_encoder_words_equal_oracle(bits):
    K, N = 32, 32  # 4 tiles
    Tg = grid_targets(100 + bits, K, N)
    words, err = tfx.encode(torch.from_numpy(Tg).to(DEV), bits)
    want, want_err = oracle.encode(Tg, K, N, bits)
    assert np.array_equal(words.cpu().numpy().view(np.uint32), want)
    assert int(err.sum()) == want_err


def test_encoder_many_tiles_sampled_and_decoded():
    # 256 x 384 at 4 bits (384 tiles, more than one per SM, ragged last round):
    # sampled tiles against the oracle, the whole weight through the layer's decoder
    K, N, bits = 256, 384, 4
    Tg = grid_targets(7, K, N)
    words, err = tfx.encode(torch.from_numpy(Tg).to(DEV), bits, max_ctas=100)
    got = words.cpu().numpy().view(np.uint32)
    tiles = (K // 16) * (N // 16)
    for t0 in (0, 151, tiles - 1):
        part, e = oracle.encode(Tg, K, N, bits, tile0=t0, ntiles=1)
        tk, tn = divmod(t0, N // 16)
        sl = slice(tn * 8 * bits, (tn + 1) * 8 * bits)
        assert np.array_equal(got[tk, sl], part[tk, sl]), t0
        assert int(err[t0]) == e
    w = tfx.Weight(words, torch.ones(K, dtype=torch.float16, device=DEV).view(torch.int16),
                   torch.ones(N, dtype=torch.float16, device=DEV).view(torch.int16), K, N, bits)
    W = tfx.debug_decode(w).float().cpu().numpy().astype(np.float64)
    assert int(((np.rint(W * 128) - Tg) ** 2).sum()) == int(err.sum())
    # 4 bits per weight: mean squared error under 1 % of the target variance
    assert float(err.sum()) / (K * N) / 128 ** 2 < 0.01 * 1.155 ** 2


def test_encoder_validation():
    t = torch.zeros((32, 32), dtype=torch.int16, device=DEV)
    for bits in (0, 9):
        with pytest.raises(tfx.TfxError):
            tfx.encode(t, bits)
    with pytest.raises(tfx.TfxError):
        tfx.encode(t, 4, scratch=torch.empty(16, dtype=torch.uint8, device=DEV))
