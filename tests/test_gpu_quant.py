"""GPU parity of the quantiser and the scale transform: bit-exact against the
oracle (E4M3 codes, exponents, packed UE8M0 words)."""
import numpy as np
import pytest
import torch

import oracle
import moe_grouped_gemm_fp8_gb300 as dg

pytestmark = pytest.mark.gpu


def _x(shape, seed, spread=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(*shape, generator=g)
    if spread:  # row-dependent magnitudes: exercises many exponents
        x = x * torch.exp(torch.randn(*shape[:-1], 1, generator=g) * 4)
    return x


@pytest.mark.parametrize("block_rows", [1, 128])
@pytest.mark.parametrize("groups,rows,cols", [(1, 300, 640), (3, 37, 128), (2, 130, 1536), (1, 1, 512)])
def test_quantize_matches_oracle(block_rows, groups, rows, cols):
    x = _x((groups, rows, cols), seed=rows * 31 + cols + block_rows)
    q_dev, sf_dev = dg.quantize_fp8(x.cuda(), block_rows, packed=False)
    q_pk, sfp_dev = dg.quantize_fp8(x.cuda(), block_rows, packed=True)
    q_dev = q_dev.view(torch.uint8).cpu().numpy()
    assert np.array_equal(q_dev, q_pk.view(torch.uint8).cpu().numpy())
    sf_dev = sf_dev.cpu().numpy()
    sfp_dev = sfp_dev.cpu().numpy()
    for g in range(groups):
        q, e, s = oracle.quantize(x[g].numpy(), block_rows)
        assert np.array_equal(q_dev[g], q), "codes differ in group %d" % g
        assert np.array_equal(sf_dev[g].astype(np.float64), s)
        assert np.array_equal(sfp_dev[g], oracle.pack_ue8m0(e, rows, block_rows))


def test_quantize_edge_values():
    # zero groups, exact power-of-two boundaries, tiny values that round to +-0
    x = torch.zeros(4, 256)
    x[1, :128] = 448.0 * 2.0 ** -5
    x[1, 5] = -448.0 * 2.0 ** -5
    x[2, :128] = torch.linspace(-1e-7, 1e-7, 128)
    x[2, 0] = 1.0
    x[3, 128:] = torch.tensor([(-1.0) ** i * 2.0 ** (i % 40 - 20) for i in range(128)])
    q_dev, sf_dev = dg.quantize_fp8(x.cuda(), 1, packed=False)
    q, e, s = oracle.quantize(x.numpy(), 1)
    assert np.array_equal(q_dev.view(torch.uint8).cpu().numpy(), q)
    assert np.array_equal(sf_dev.cpu().numpy().astype(np.float64), s)


@pytest.mark.parametrize("block_rows,groups,mn,k", [(1, 1, 300, 640), (128, 3, 200, 1536), (1, 2, 7, 128)])
def test_transform_sf_matches_oracle_pack(block_rows, groups, mn, k):
    rng = np.random.default_rng(mn + k)
    mb = (mn + block_rows - 1) // block_rows
    e = rng.integers(-127, 128, size=(groups, mb, k // 128)).astype(np.int32)
    sf = torch.from_numpy(np.ldexp(1.0, e).astype(np.float32)).cuda()
    got = dg.transform_sf_into_required_layout(sf, mn, k, block_rows).cpu().numpy()
    assert np.array_equal(got, oracle.pack_ue8m0(e, mn, block_rows))
    st, _ = dg.get_device_error()
    assert st == 0


def test_transform_sf_flags_non_power_of_two():
    dg.get_device_error()  # clear
    sf = torch.ones(1, 4, 2).cuda()
    sf[0, 2, 1] = 3.0
    got = dg.transform_sf_into_required_layout(sf, 4, 256, 1).cpu().numpy().view(np.uint32)
    st, word = dg.get_device_error()
    assert st == 8 and (word & 0xFF) == 8  # DG_ERR_DEVICE_BAD_SCALE
    assert got.shape == (1, 1, 4)
    assert ((got[0, 0, 2] >> 8) & 0xFF) == 127 + 2  # 3.0 rounded up to 4.0
    assert (got[0, 0, 0] & 0xFFFF) == 0x7F7F
