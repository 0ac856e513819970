import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built library")
    config.addinivalue_line("markers", "slow: long-running statistical or full-size case")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


class _BigWeights:
    """Full-size LM-head weights, generated once per session: host bits, a
    device copy and (lazily) the float64 copy the oracle multiplies with."""

    def __init__(self, vocab, hidden):
        import numpy as np
        import torch
        from speculative_decoding_verify_row_gb300 import synth
        self.vocab, self.hidden = vocab, hidden
        self.bits = synth.weights(vocab, hidden)
        self.dev = torch.from_numpy(self.bits.view(np.int16)).cuda()
        self._w64 = None

    def oracle_logits(self, act):
        """float64 oracle logits [R, V] (the oracle's projection, with the
        float64 weights cached across calls)."""
        import numpy as np
        from oracle import verify as ov
        if self._w64 is None:
            self._w64 = ov.bf16_bits_to_f32(self.bits).astype(np.float64)
        return np.asarray(act, np.float32).astype(np.float64) @ self._w64.T


@pytest.fixture(scope="session")
def big_weights_4096():
    return _BigWeights(151936, 4096)


@pytest.fixture(scope="session")
def big_weights_5120():
    return _BigWeights(151936, 5120)


def pytest_terminal_summary(terminalreporter):
    mod = sys.modules.get("test_gpu_window")
    if mod is not None and mod.END_TO_END["windows"]:
        e = mod.END_TO_END
        terminalreporter.write_line(
            f"fused windows compared end to end with the oracle: {e['compared']} of "
            f"{e['windows']} (the rest had a float32 near-tie that reorders a pool)")
