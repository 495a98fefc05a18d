"""The timeout path on the GPU: a wait that nothing satisfies ends the kernel with a status.

The test hook ``debug_flags = 1`` starts the producer end of the SMEM ring at
phase 0 instead of 1 — the "opposite initial phases" mistake that "GEMM III"
warns deadlocks the pipeline.  Every role then waits on a barrier that nothing
will complete; each wait has a short limit, after which the kernel records the
failure in its status word and returns.  The context must stay usable: a normal
GEMM right afterwards must be correct.  No trap, no fault, no unbounded spin.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

TIMEOUT = -7


# (cta_group, consumers, block_n, block_m, cluster_k): the CTA pair, a single CTA, two
# consumers, narrow, tiny and thin tiles, and narrow and tiny tiles with K split across clusters
# of 2, 4 and 8 CTAs (there every CTA still reaches the cluster barrier after its roles gave up)
VARIANTS = [(2, 1, 0, 0, 0), (1, 1, 0, 0, 0), (2, 2, 0, 0, 0), (1, 1, 64, 128, 1), (1, 1, 64, 128, 2),
            (1, 1, 64, 64, 1), (1, 1, 64, 64, 4), (1, 1, 64, 64, 8), (1, 1, 16, 64, 1)]


@pytest.mark.parametrize("cg,consumers,bn,bm,ks", VARIANTS,
                         ids=["pair", "single", "pair-2consumers", "narrow", "narrow-k2", "tiny", "tiny-k4",
                              "tiny-k8", "thin"])
def test_deadlocked_ring_times_out_and_context_survives(gpu_lib, cg, consumers, bn, bm, ks):
    w = si.WORKLOADS["ktile_grid_256x256x512"]
    A, B = w.operands()
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    D = torch.zeros((w.M, w.N), dtype=torch.float16, device="cuda")
    shape = dict(cta_group=cg, consumers=consumers, block_n=bn, block_m=bm, cluster_k=ks)
    bad = gpu_lib.Options(**shape, debug_flags=1, timeout_ns=100_000_000)  # 0.1 s a wait
    gpu_lib.gemm_f16_nt(dA, dB, D, options=bad)
    status, info = gpu_lib.last_device_status()
    assert status == TIMEOUT, gpu_lib.status_string(status)
    # every role waits from the start on a barrier nothing completes; whichever
    # limit runs out first is recorded (producer 1, MMA issuer 2, epilogue 3)
    assert info >> 56 in (1, 2, 3)
    # a later, correct launch on the same context works and leaves the status clear
    D2 = gpu_lib.gemm_f16_nt(dA, dB, options=gpu_lib.Options(**shape))
    assert gpu_lib.last_device_status()[0] == 0
    got = D2.cpu().numpy().astype(np.float64)
    ref = oracle.gemm_f16_nt(A, B).view(np.float16).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2.0 ** -9 * np.abs(ref) + 1e-3)
