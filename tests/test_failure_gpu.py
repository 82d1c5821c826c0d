"""Failure reporting on the GPU without faulting or hanging it.

A plan's wait-test hook makes every ring slot wait for 16 bytes that never
arrive; with a 20 ms wait limit the kernel's bounded waits run out, the kernel
records the failure in the plan's error word, unwinds (lets copies land, drains
MMAs, frees TMEM) and exits.  The host must see GEMM_ERR_DEVICE_TIMEOUT from
gemm_plan_check, and the same plan must then compute a correct result.
"""
import pytest
import torch

import dense_gemm_hgemm_gb300 as g
from dense_gemm_hgemm_gb300 import inputs

import parity_util as pu

pytestmark = pytest.mark.gpu

CONFIGS = [
    ("one_sm", (256, 320, 512), {"block_n": 128}),
    ("workspace_split", (128, 128, 1024), {"block_n": 64, "split_k": 4}),
    ("cluster_split", (128, 128, 1024), {"block_n": 64, "split_k": 4, "split_mode": 1}),
    ("sm_pair", (512, 512, 512), {"block_n": 256, "cta_pair": 1}),
    ("sm_pair_split", (512, 512, 1024), {"block_n": 256, "cta_pair": 1, "split_k": 4,
                                         "split_mode": 1}),
    ("multicast", (256, 512, 512), {"block_n": 64, "multicast": 4}),
    ("two_kblock_slots", (256, 512, 1024), {"block_n": 64, "kblocks_per_stage": 2}),
    ("sm_pair_two_kblock_slots", (512, 512, 1024), {"block_n": 256, "cta_pair": 1,
                                                    "kblocks_per_stage": 2}),
]


@pytest.mark.parametrize("name,shape,cfg", CONFIGS, ids=[c[0] for c in CONFIGS])
def test_wait_timeout_is_reported_and_context_survives(gemm_lib, name, shape, cfg):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "f16")
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    with g.Plan(M, N, K, "f16", cfg) as plan:
        plan.set_timeout(20_000_000)          # 20 ms
        plan.set_wait_test(16)
        plan.run(dA, dB, C)
        with pytest.raises(g.GemmError) as e:
            plan.check()
        assert e.value.status == 9            # GEMM_ERR_DEVICE_TIMEOUT
        plan.set_wait_test(0)
        plan.set_timeout(0)
        plan.run(dA, dB, C)
        plan.check()                          # error word was cleared; normal run is clean
    pu.check_full(A, B, "f16", C, "after timeout: " + name)


def test_wait_test_hook_validates(gemm_lib):
    with g.Plan(128, 128, 64, "f16") as plan:
        for bad in (7, 8192):
            with pytest.raises(g.GemmError):
                plan.set_wait_test(bad)
