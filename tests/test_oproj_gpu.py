"""GPU parity of the output projection (kda_o_proj, the library's tcgen05 GEMM: bf16
operands, fp32 accumulation) against the oracle's fp64 matmul of the same bf16 inputs:
ragged small cases in fp32 and bf16 output on both tile widths, the decode shape of the
layer (256 x 12288 -> 7168) element by element and the prefill shape on sampled outputs.  Tolerance: fp32 accumulation over K terms of unit-scale products
(max|diff| / rms 1e-4); bf16 outputs add one rounding per element (2^-8 relative)."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_gated_gb300 as kda
import oracle
from tests.gpu_helpers import rel_err

pytestmark = pytest.mark.gpu


def _data(rows, K, N, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    y = torch.randn((rows, K), generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn((N, K), generator=g, device="cuda") * K ** -0.5).to(torch.bfloat16)
    return y, w


def _check(out, ref, out_dtype):
    if out_dtype == torch.float32:
        assert rel_err(out, ref) <= 1e-4
    else:  # one bf16 rounding of each output (half an ulp: 2^-9 relative) on top of fp32 accumulation
        rms = float(np.sqrt(np.mean(ref * ref)))
        assert np.all(np.abs(out.double().cpu().numpy() - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-4 * rms)


@pytest.mark.parametrize("rows,K,N", [(1, 512, 1024), (129, 512, 1024), (300, 256, 640), (5, 576, 512),
                                      (700, 256, 7168),  # 256-row tiles, several per pair
                                      (1100, 256, 7168),  # 512-row tiles, the last one's upper half empty
                                      (1500, 256, 7168)])  # 512-row tiles, the last one ending in its upper half
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_tile_edges(rows, K, N, out_dtype):
    """Row counts that end inside a token tile: the pair kernels (out_features a multiple of
    256; K split over two pairs for at most 256 rows and an even count of 64-wide K slices,
    else the persistent form: 256-row tiles at 700 rows, 512-row tiles once every pair still
    gets one, at 1100 and 1500 rows) and the single-CTA kernel (640 features)."""
    y, w = _data(rows, K, N, rows)
    out = kda.o_proj(y, w, out_dtype=out_dtype)
    torch.cuda.synchronize()
    _check(out, oracle.o_proj(y.float().cpu().numpy(), w.float().cpu().numpy()), out_dtype)


def test_decode_shape_every_element():
    """The decode batch of the layer: 256 rows x 12288 -> 7168, every output element."""
    y, w = _data(256, 12288, 7168, 11)
    out = kda.o_proj(y, w, out_dtype=torch.float32)
    torch.cuda.synchronize()
    kda.device_status()
    assert rel_err(out, oracle.o_proj(y.float().cpu().numpy(), w.float().cpu().numpy())) <= 1e-4


def test_unsupported_feature_counts():
    y, w = _data(4, 1000, 768, 3)
    with pytest.raises(kda.KDAError):
        kda.o_proj(y, w)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_small_ragged(out_dtype):
    y, w = _data(37, 1024, 768, 0)
    out = kda.o_proj(y, w, out_dtype=out_dtype)
    torch.cuda.synchronize()
    ref = oracle.o_proj(y.float().cpu().numpy(), w.float().cpu().numpy())
    if out_dtype == torch.float32:
        assert rel_err(out, ref) <= 1e-4
    else:  # one bf16 rounding of each output (half an ulp: 2^-9 relative) on top of fp32 accumulation
        rms = float(np.sqrt(np.mean(ref * ref)))
        assert np.all(np.abs(out.double().cpu().numpy() - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-4 * rms)


@pytest.mark.parametrize("rows", [256, 8192])
def test_layer_shape_sampled(rows):
    y, w = _data(rows, 12288, 7168, 1 + rows)
    out = kda.o_proj(y, w, out_dtype=torch.float32)
    torch.cuda.synchronize()
    cols = np.sort(np.random.default_rng(rows).choice(7168, 64, replace=False))
    rsel = np.sort(np.random.default_rng(rows + 1).choice(rows, min(rows, 256), replace=False))
    ref = oracle.o_proj(y[torch.from_numpy(rsel).cuda()].float().cpu().numpy(),
                        w[torch.from_numpy(cols).cuda()].float().cpu().numpy())
    got = out[torch.from_numpy(rsel).cuda()][:, torch.from_numpy(cols).cuda()]
    assert rel_err(got, ref) <= 1e-4
