"""The tensor-core kernels' abort path, exercised without faulting anything:
a short limit on the MMA issuer's stage wait (a diagnostic of the C ABI)
makes that wait run out on the first stage. The kernel must record
NF4_ERR_DEVICE_TIMEOUT with its site (kernel, role = MMA issuer, CTA), let
its copies and MMAs in flight finish, free its tensor memory and return; the
next call with the default limit must then be correct. Every other wait
keeps its full limit, so nothing can be left waiting."""
import numpy as np
import pytest
import torch

import dequant_gemm_gb300 as nf4
from dequant_gemm_gb300 import workloads as wl
from oracle import nf4_oracle as o

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TIMEOUT = 7
KERNEL_FWD, KERNEL_DX, ROLE_MMA = 2, 3, 2


@pytest.mark.parametrize("dx", [False, True], ids=["fwd", "dx"])
@pytest.mark.parametrize("M", [40, 300], ids=["single", "pair"])
def test_short_mma_wait_takes_the_abort_path_and_recovers(M, dx):
    W = wl.weight(520, 1024, seed=70).numpy()
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV))
    A = wl.activations(M, 520 if dx else 1024, seed=M + 71, std=0.01 if dx else 1.0).to(DEV)
    fn = nf4.nf4_matmul_bwd_dx if dx else nf4.nf4_matmul_fwd
    assert nf4.nf4_poll_device_status_site() == (0, 0)
    nf4.nf4_set_mma_wait_limit(200)
    try:
        fn(A, q)
        status, site = nf4.nf4_poll_device_status_site()
    finally:
        nf4.nf4_set_mma_wait_limit(0)
    assert status == TIMEOUT, status
    u = site & 0xffffffff
    assert u >> 28 == (KERNEL_DX if dx else KERNEL_FWD), nf4.describe_site(site)
    assert (u >> 24) & 15 == ROLE_MMA, nf4.describe_site(site)
    # the same call again, default limit: correct and no status
    out = fn(A, q).cpu().numpy()
    assert nf4.nf4_poll_device_status_site() == (0, 0)
    Wh = o.dequantize(*o.quantize(W), 520, 1024)
    ref = o.matmul_bwd_dx(A.float().cpu().numpy(), Wh) if dx else o.matmul_fwd(A.float().cpu().numpy(), Wh)
    assert o.rel_frobenius(out, ref) <= 2e-3 and o.max_rel_to_max(out, ref) <= 5e-3
