"""The measurement hooks.  The tensor-pipe rate probe (mma_rate): every CTA
finishes its MMAs and reports a dense bf16 rate per SM per clock within the
data-sheet figure for this architecture, 8192 FLOP per SM per clock (4096
bf16 multiply-adds), which it must not exceed.  The clock log
(gemm_clock_log): the GEMM's CTA 0 reports clock ticks and nanoseconds whose
ratio is an SM clock this GPU can run at, and nothing once it is turned off."""
import pytest
import torch

from stage_software_pipelining_gb300 import build as gemm_build
from stage_software_pipelining_gb300 import gemm as G

pytestmark = pytest.mark.gpu

NOMINAL_FLOP_PER_CLK = 8192


@pytest.fixture(scope="module", autouse=True)
def library(gpu):
    gemm_build.build()
    G.load_library()


def test_rate_on_every_sm():
    r = G.mma_rate(n_mma=8192)
    assert r["ctas"] == torch.cuda.get_device_properties(0).multi_processor_count
    assert r["cycles_min"] > 0
    rate = r["flop_per_clk_per_sm"]
    assert 0.9 * NOMINAL_FLOP_PER_CLK <= rate <= 1.01 * NOMINAL_FLOP_PER_CLK, r
    # the SMs agree: one slow SM would show as a spread of clocks
    assert r["cycles_max"] <= 1.05 * r["cycles_min"], r


def test_pair_rate_on_every_tpc():
    """The CTA-pair instruction of the 256-row tiles runs at the same rate
    per SM as the one-CTA one."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    r = G.mma_rate(n_mma=8192, pair=True)
    assert r["ctas"] == sms - sms % 2 and r["pair"]
    assert r["cycles_min"] > 0
    rate = r["flop_per_clk_per_sm"]
    assert 0.9 * NOMINAL_FLOP_PER_CLK <= rate <= 1.01 * NOMINAL_FLOP_PER_CLK, r
    assert r["cycles_max"] <= 1.05 * r["cycles_min"], r
    one = G.mma_rate(n_mma=64, ctas=2, pair=True)
    assert one["cycles_min"] > 0


@pytest.mark.parametrize("n_mma", [1, 3, 4096])
def test_small_counts_and_one_cta(n_mma):
    r = G.mma_rate(n_mma=n_mma, ctas=1)
    assert r["cycles_min"] > 0
    if n_mma >= 4096:
        assert r["flop_per_clk_per_sm"] <= 1.01 * NOMINAL_FLOP_PER_CLK, r


def test_rejects_more_ctas_than_sms():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    with pytest.raises(G.GemmError):
        G.mma_rate(n_mma=16, ctas=sms + 1)


@pytest.mark.parametrize("tile", [G.TILE_128x128, G.TILE_128x256, G.TILE_256x256_2SM,
                                  G.TILE_256x512_2SM, "simt"])
def test_clock_log_of_the_gemm(tile):
    gen = torch.Generator().manual_seed(7)
    dt = torch.float32 if tile == "simt" else torch.bfloat16
    A = (torch.rand(2048, 2048, generator=gen) - 0.5).to(dt).cuda()
    B = (torch.rand(2048, 2048, generator=gen) - 0.5).to(dt).cuda()
    if tile == "simt":
        tile = G.SIMT_FRAGMENTS_DOUBLE
    C = torch.zeros(2048, 2048, device="cuda")
    log = torch.zeros(2, dtype=torch.int64, device="cuda")
    G.clock_log(log)
    try:
        for _ in range(5):
            G.gemm(A, B, C, 1.0, 0.0, stages=3, tile=tile)
        torch.cuda.synchronize()
    finally:
        G.clock_log(None)
    ticks, ns = log.tolist()
    assert ticks > 0 and ns > 0
    mhz = ticks * 1000.0 / ns
    assert 300.0 <= mhz <= 2200.0, mhz
    # off: later launches add nothing
    G.gemm(A, B, C, 1.0, 0.0, stages=3, tile=tile)
    torch.cuda.synchronize()
    assert log.tolist() == [ticks, ns]
    with pytest.raises(ValueError):
        G.clock_log(torch.zeros(2, dtype=torch.int32, device="cuda"))
