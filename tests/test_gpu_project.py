"""GPU parity of the verify projection (both paths) against the fp64 oracle,
and the row-count invariance the pages require ("Speculative decoding on
RDNA" §02: multi-row verify projections sum in the single-row order)."""
import numpy as np
import pytest
import torch

from oracle import verify as ov
from speculative_decoding_verify_row_gb300 import binding as vb, synth
from gpu_common import require_gpu, dev_weight, dev, project, assert_logits_close

pytestmark = pytest.mark.gpu
PATHS = [vb.VR_PATH_TC, vb.VR_PATH_FFMA, vb.VR_PATH_TC_BATCH]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("path", PATHS)
def test_tiny_config(path):
    W = synth.weights(4096, 256)
    A = synth.activations(4, 256, 0)
    got = project(dev_weight(W), A, path).cpu().numpy()
    assert_logits_close(got, ov.project(W, A))


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("H,V", [(520, 5000), (8, 300), (4104, 777), (64, 128), (1000, 129)])
@pytest.mark.parametrize("R", [1, 5, 33])
def test_ragged_shapes(path, H, V, R):
    rng = np.random.default_rng(H * 7 + V + R)
    W = synth.f32_to_bf16_bits(rng.standard_normal((V, H), dtype=np.float32) * np.float32(0.05))
    A = rng.standard_normal((R, H), dtype=np.float32)
    got = project(dev_weight(W), A, path).cpu().numpy()
    assert_logits_close(got, ov.project(W, A))


@pytest.mark.parametrize("path", PATHS)
def test_row_bits_do_not_depend_on_row_count(path):
    rng = np.random.default_rng(11)
    V, H = 3000, 1032
    W = dev_weight(synth.f32_to_bf16_bits(rng.standard_normal((V, H), dtype=np.float32) * np.float32(0.03)))
    A = rng.standard_normal((40, H), dtype=np.float32)
    full = project(W, A, path).cpu().numpy().view(np.uint32)
    for R in list(range(1, 33)) + [33, 40]:
        part = project(W, A[:R], path).cpu().numpy().view(np.uint32)
        assert np.array_equal(part, full[:R]), R
    # a row alone, and the same row next to unrelated rows, in any slot
    for r in (0, 7, 31, 39):
        alone = project(W, A[r:r + 1], path).cpu().numpy().view(np.uint32)
        assert np.array_equal(alone[0], full[r])
        other = rng.standard_normal((25, H), dtype=np.float32)
        other[13] = A[r]
        mixed = project(W, other, path).cpu().numpy().view(np.uint32)
        assert np.array_equal(mixed[13], full[r])


@pytest.fixture(scope="module")
def big_weight():
    W = synth.weights(151936, 4096)
    return W, dev_weight(W)


@pytest.mark.parametrize("path", PATHS)
def test_full_size_sampled_rows(big_weight, path):
    """H 4096 x V 151936 at 25 rows (the tree size), checked on 3000 sampled
    vocab rows (plus both ends) against the oracle, and 1-row vs 25-row bit
    identity over the whole vocabulary."""
    W, Wd = big_weight
    A = synth.activations(25, 4096, 3)
    got = project(Wd, A, path)
    rng = np.random.default_rng(5)
    cols = np.unique(np.concatenate([rng.integers(0, 151936, 3000), [0, 1, 151934, 151935]]))
    assert_logits_close(got[:, torch.from_numpy(cols).cuda()].cpu().numpy(),
                        ov.project_columns(W, A, cols))
    one = project(Wd, A[7:8], path)
    assert torch.equal(one[0].view(torch.int32), got[7].view(torch.int32))


@pytest.mark.parametrize("path", PATHS)
def test_row_bits_across_row_groups(path):
    """More rows than one group of any path (300 > 256 > 32 > 8): every row
    equals the same row computed alone, and matches the oracle."""
    rng = np.random.default_rng(12)
    V, H = 1100, 520
    Wb = synth.f32_to_bf16_bits(rng.standard_normal((V, H), dtype=np.float32) * np.float32(0.03))
    W = dev_weight(Wb)
    A = rng.standard_normal((300, H), dtype=np.float32)
    full = project(W, A, path)
    assert_logits_close(full.cpu().numpy(), ov.project(Wb, A))
    full = full.cpu().numpy().view(np.uint32)
    for r in (0, 31, 32, 255, 256, 299):
        alone = project(W, A[r:r + 1], path).cpu().numpy().view(np.uint32)
        assert np.array_equal(alone[0], full[r]), r


@pytest.mark.parametrize("path", PATHS)
def test_unaligned_activations(path):
    """Activations at an address that is not 16-byte aligned give the same
    bits as an aligned copy."""
    rng = np.random.default_rng(17)
    V, H, R = 2000, 520, 5
    Wb = synth.f32_to_bf16_bits(rng.standard_normal((V, H), dtype=np.float32) * np.float32(0.05))
    W = dev_weight(Wb)
    A = rng.standard_normal((R, H), dtype=np.float32)
    aligned = torch.from_numpy(A).cuda()
    buf = torch.empty(R * H + 1, dtype=torch.float32, device="cuda")
    buf[1:] = aligned.reshape(-1)
    shifted = buf[1:].view(R, H)
    assert shifted.data_ptr() % 16 != 0
    outs = []
    for act in (aligned, shifted):
        lg = torch.empty((R, V), dtype=torch.float32, device="cuda")
        vb.verify_project(W, act, lg, vb.workspace(R, H, V), path=path)
        torch.cuda.synchronize()
        outs.append(lg.cpu().numpy().view(np.uint32))
    assert np.array_equal(outs[0], outs[1])
    assert_logits_close(outs[1].view(np.float32), ov.project(Wb, A))
