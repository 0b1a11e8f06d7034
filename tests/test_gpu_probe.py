"""The dense FP8 tensor-core probe runs its MMAs: the first CTA's accumulator
element (0, 0) equals 32 * iters exactly (every operand element is 0.5, so
each of the 4 * iters K=32 steps adds 32 * 0.25), and the reported FLOP count
is 2 * 128 * 256 * 32 per MMA on every SM."""

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("iters", [1, 7, 1000])
def test_probe_accumulates_every_mma(iters):
    import sparse_attention_indexer_nvfp4_gb300 as idx

    check = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flops = idx.idx_fp8_mma_probe(iters, check, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert float(check.item()) == 32.0 * iters
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert flops == 2.0 * 128 * 256 * 32 * 4 * iters * sms
