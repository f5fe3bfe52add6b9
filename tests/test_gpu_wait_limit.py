"""Failure detection without a GPU fault: every wait inside the kernel is
bounded.  With the limit set to 0 the first wait that is not already over
expires; the kernel must then abandon the launch cleanly (drain its copies and
MMAs, free tensor memory), report XS_ERR_DEVICE_TIMEOUT through the device error
word, and leave the CUDA context usable for the next, correct, launch."""
import math

import numpy as np
import pytest

import dit_inputs as di
from _parity import abs_bits, assert_close, bits_to_torch, torch_to_f64

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def xs():
    from conftest import build_library
    build_library()
    import dit_attention_ulysses_gb300 as xs
    return xs


def test_expired_wait_is_reported_and_context_survives(xs, monkeypatch):
    import oracle
    w = di.Workload("wl", B=1, H=4, S=1024, D=128, P=4, scale=1 / math.sqrt(128))
    qb, kb, vb = di.random_qkv(w)
    q, k, v = (bits_to_torch(x) for x in (qb, kb, vb))
    outs = [torch.zeros((1, 256, 4, 128), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    assert xs.xs_attn_get_device_error() == xs.XS_OK

    monkeypatch.setenv("XSATTN_WAIT_TIMEOUT_NS", "0")
    xs.xs_attn_a2a_fwd(q, k, v, outs, w.scale)          # the launch itself succeeds
    code, rec = xs.xs_attn_get_device_error_info()
    assert code == xs.XS_ERR_DEVICE_TIMEOUT
    # the record names the wait: a CTA of the 32-tile grid, one of its 12 warps,
    # an mbarrier address in shared memory, a parity and the piece it waited in
    assert rec["kind"] == 1
    assert 0 <= rec["cta"] < 32 and 0 <= rec["warp"] < 12 and 0 <= rec["lane"] < 32
    assert 0 < rec["site"] < 232448 and rec["detail0"] in (0, 1) and rec["detail1"] >= 0
    assert xs.xs_attn_get_device_error_info() == (xs.XS_OK, {k: 0 for k in rec})   # cleared
    monkeypatch.delenv("XSATTN_WAIT_TIMEOUT_NS")

    torch.cuda.synchronize()                            # the context is intact
    xs.xs_attn_a2a_fwd(q, k, v, outs, w.scale)
    assert xs.xs_attn_get_device_error() == xs.XS_OK
    ref = oracle.attention_a2a(qb, kb, vb, w.scale, w.P)
    mass = oracle.attention_a2a(qb, kb, abs_bits(vb), w.scale, w.P)
    assert_close(np.stack([torch_to_f64(o) for o in outs]), ref, mass, "after timeout")
