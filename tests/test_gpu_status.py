"""Failure path on the GPU without a fault: a kernel whose wait nothing
completes must give up after its time limit and report GEMMA3_ERR_TIMEOUT,
leaving the context usable; invalid arguments are refused before launch."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from transformer_attention_gb300.build import build
    build()


def test_bounded_wait_reports_timeout_and_context_survives():
    import transformer_attention_gb300 as G3
    from transformer_attention_gb300 import _lib as L
    rc = G3.gemma3_selftest_wait_timeout(50_000_000)   # 50 ms
    assert rc == L.GEMMA3_ERR_TIMEOUT
    assert G3.gemma3_last_device_status() == 0x1000 + 99
    # the status word was cleared and the context still works
    assert G3.gemma3_attn_check_status() == 0
    a = torch.ones(256, 64, dtype=torch.bfloat16, device="cuda")
    c = G3.linear(a, a, out_dtype=torch.float32)
    assert G3.gemma3_attn_check_status() == 0
    assert torch.all(c == 64)


def test_invalid_arguments_refused_on_gpu():
    import transformer_attention_gb300 as G3
    x = torch.zeros(1, 64, 1152, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(G3.Gemma3Error):
        G3.gemma3_flash_attention(x, x, x, 256, x, 0, None, 1, 64, 8, 1, 256, 0)   # G = 8
    with pytest.raises(G3.Gemma3Error):
        G3.gemma3_linear(x, 1152, x, 1152, x, 1152, 64, 64, 1152, 0, 9)            # bad dtype
