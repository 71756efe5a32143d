"""GPU tests of the library's failure detection, made to happen without a fault: the
first-line waits on copies from global memory (decode step, short convolution, the fused
prefill kernel) get a bound of zero polls (kda_set_wait_limit), so every such wait gives
up at once while its copy is still in flight.  The kernel then lets
the copy land (that wait keeps its full bound), writes NaN into every output it was
responsible for and counts the event; kda_device_status reports KDA_ERR_TIMEOUT once and
clears the count, and the next call on the same context computes correctly.  No test
here faults, traps or hangs the GPU."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_gated_gb300 as kda
import oracle
from kimi_delta_attention_gated_gb300.inputs import make_conv_inputs, make_inputs
from tests.gpu_helpers import FP32_TOL, PARITY, np32, oracle_run, rel_err
from tests.test_parity_gpu import decode_inputs, decode_oracle

pytestmark = pytest.mark.gpu
TIMEOUT = 4


@pytest.fixture(scope="module", autouse=True)
def built():
    from kimi_delta_attention_gated_gb300 import build
    build.build()


@pytest.fixture()
def zero_wait_limit():
    kda.device_status()  # nothing pending from earlier tests
    kda.set_wait_limit(0)
    try:
        yield
    finally:
        kda.set_wait_limit(None)


def expect_timeout():
    with pytest.raises(kda.KDAError) as e:
        kda.device_status()
    assert e.value.status == TIMEOUT
    kda.device_status()  # the counters were cleared: a second check passes


def test_decode_timeout_poisons_every_unit_it_owned(zero_wait_limit):
    """4 x 100 = 400 units over a grid of at most 2 CTAs per SM: on a 152-SM GPU most
    CTAs own two units, so the second (never reached) unit must be poisoned too.  The
    state is updated in place, where an unwritten unit would keep its old, valid-looking
    state."""
    d = decode_inputs(B=4, H=100)
    state = d["initial_state"].clone()
    o, s, y = kda.recurrent_step(d["q"], d["k"], d["v"], d["g"], d["beta"], state, gate=d["gate"],
                                 norm_w=d["norm_w"], eps=d["eps"], state_out=state)
    expect_timeout()
    assert torch.isnan(s).all() and torch.isnan(o).all() and torch.isnan(y).all()


def test_decode_after_a_timeout_is_correct():
    """The context stays usable: with the default bound the same step matches the oracle."""
    kda.set_wait_limit(0)
    try:
        d = decode_inputs(B=2, H=3)
        kda.recurrent_step(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"].clone(),
                           gate=d["gate"], norm_w=d["norm_w"], eps=d["eps"])
        expect_timeout()
    finally:
        kda.set_wait_limit(None)
    d = decode_inputs(B=2, H=3)
    o, s, y = kda.recurrent_step(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                                 gate=d["gate"], norm_w=d["norm_w"], eps=d["eps"])
    kda.device_status()
    oo, so, yo = decode_oracle(d)
    assert rel_err(o, oo) <= FP32_TOL
    assert rel_err(s, so) <= FP32_TOL
    assert rel_err(y, yo) <= FP32_TOL


def test_short_conv_timeout_poisons_outputs_and_states(zero_wait_limit):
    """Every tile wait gives up: y is NaN everywhere and so is the carried state of both
    sequences (their last tokens lie in poisoned tiles)."""
    d = make_conv_inputs(device="cuda", B=2, T=70, D=256, W=4, state=True)
    y, s = kda.short_conv(d["x"], d["weight"], None, d["conv_state"], out_dtype=torch.float32)
    expect_timeout()
    assert torch.isnan(y).all() and torch.isnan(s).all()
    kda.set_wait_limit(None)
    y, s = kda.short_conv(d["x"], d["weight"], None, d["conv_state"], out_dtype=torch.float32)
    kda.device_status()
    yo, so = oracle.short_conv(np32(d["x"]), np32(d["weight"]), None, np32(d["conv_state"]))
    assert rel_err(y, yo) <= FP32_TOL
    assert rel_err(s, so) <= FP32_TOL


@pytest.mark.parametrize("norm", [False, True])
def test_prefill_timeout_poisons_every_unit(zero_wait_limit, norm):
    """The fused tensor-core prefill: every CTA's first g-tile wait gives up, the CTA lets
    its V and g copies land, and o, y and the final state (updated in place, where an
    unwritten unit would keep its old, valid-looking state) hold NaN for every unit; two
    sequences of different lengths, one with a ragged last chunk."""
    d = make_inputs("long", device="cuda", lengths=[150, 64], H=3)
    state = 0.02 * torch.randn((2, 3, 128, 128), device="cuda")
    kw = dict(gate=d["gate"], norm_w=d["norm_w"], eps=d["eps"]) if norm else {}
    res = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], state, scale=d["scale"], mode="tensor",
                        cu_seqlens=d["cu_seqlens"], final_state=state, **kw)
    expect_timeout()
    for t in res:
        assert torch.isnan(t).all()


def test_prefill_after_a_timeout_is_correct():
    """After the poisoned call, the same prompt with the default bound matches the oracle."""
    d = make_inputs("prefill", device="cuda", T=200, H=2)
    kda.set_wait_limit(0)
    try:
        kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"], mode="tensor")
        expect_timeout()
    finally:
        kda.set_wait_limit(None)
    o, s = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"], mode="tensor")
    kda.device_status()
    oo, so = oracle_run(d)
    assert rel_err(o, oo) <= PARITY
    assert rel_err(s, so) <= PARITY


def test_status_is_clean_after_normal_work():
    d = decode_inputs(B=3, H=4)
    kda.recurrent_step(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], gate=d["gate"],
                       norm_w=d["norm_w"], eps=d["eps"])
    kda.device_status()
