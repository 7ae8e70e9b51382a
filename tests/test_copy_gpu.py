"""GPU parity of the streaming-copy counter-example (pipelined_copy) against
its oracle definition (a byte-for-byte copy): bit-exact for every stage count,
sizes from one 16-byte chunk to a ragged multi-wave array, with canaries
behind the copied range."""
import numpy as np
import pytest
import torch

import oracle
from stage_software_pipelining_gb300 import build as gemm_build
from stage_software_pipelining_gb300 import gemm as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library(gpu):
    gemm_build.build()
    G.load_library()


@pytest.mark.parametrize("stages", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("n_bytes", [16, 4096, (1 << 20) + 48, (64 << 20) + 16 * 1001])
def test_copy_is_bit_exact(stages, n_bytes):
    gen = torch.Generator().manual_seed(n_bytes + stages)
    host = torch.randint(0, 256, (n_bytes,), generator=gen, dtype=torch.uint8)
    src = host.cuda()
    canary = 0xA5
    dst_buf = torch.full((n_bytes + 4096,), canary, dtype=torch.uint8, device="cuda")
    G.pipelined_copy(dst_buf[:n_bytes], src, stages)
    torch.cuda.synchronize()
    got = dst_buf.cpu().numpy()
    expect = oracle.copy_bytes(host.numpy())
    assert np.array_equal(got[:n_bytes], expect)
    assert np.all(got[n_bytes:] == canary), "a write landed past the copied range"
