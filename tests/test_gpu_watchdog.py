"""GPU watchdog: a dropped producer arrival makes a bounded wait expire; the
call reports GEMMRELU_ERR_TIMEOUT through gemm_relu_status and the context
stays usable.  No fault, trap or hang: the wait gives up after 20 ms."""
import numpy as np
import pytest

import tiled_tensor_core_03_gb300 as gr
from tiled_tensor_core_03_gb300 import inputs

from gpu_common import abs_dot, assert_parity, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _restore():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gr.status()
    yield
    gr.gemm_relu_debug_set(0, 0)
    gr.status()


@pytest.mark.parametrize("kind", ["tma", "lsu", "gemv", "splitk_cluster", "splitk_two_stage"])
def test_dropped_arrival_times_out_and_recovers(orc, kind):
    shapes = {"tma": (256, 512, 256), "lsu": (255, 509, 250), "gemv": (4, 2048, 2048),
              "splitk_cluster": (16, 1024, 2048), "splitk_two_stage": (16, 1024, 2048)}
    M, N, K = shapes[kind]
    A, B = inputs.make(M, N, K, seed=8)
    a, b = dev(A), dev(B)
    split = kind.startswith("splitk")
    if kind == "splitk_two_stage":
        gr.gemm_relu_debug_force_split(gr.SPLIT_TWO_STAGE)
    try:
        gr.gemm_relu_debug_set(1, 20_000_000)
        if split:
            gr.gemm_relu_splitk(a, b, 4)
        else:
            gr.gemm_relu(a, b)
        assert gr.status() == gr.ERR_TIMEOUT
        assert gr.status() == gr.OK            # reading clears the word
        gr.gemm_relu_debug_set(0, 0)
        c = gr.gemm_relu_splitk(a, b, 4) if split else gr.gemm_relu(a, b)
        assert gr.status() == gr.OK
    finally:
        gr.gemm_relu_debug_force_split(gr.SPLIT_AUTO)
    assert_parity(host(c), orc.gemm_relu_f16(A, B), abs_dot(A, B), K, kind)


@pytest.mark.parametrize("kernel", [1, 3])
def test_streamk_dropped_arrival_times_out_and_recovers(orc, kernel):
    M, N, K = 2304, 2304, 4096
    A, B = inputs.make(M, N, K, seed=9)
    a, b = dev(A), dev(B)
    gr.gemm_relu_debug_force_kernel(kernel)
    try:
        assert gr.gemm_relu_f16_streamk_workspace_bytes(M, N, K) > 0
        ws = gr.streamk_workspace(M, N, K)
        gr.gemm_relu_debug_set(1, 20_000_000)
        gr.gemm_relu_streamk(a, b, workspace=ws)
        assert gr.status() == gr.ERR_TIMEOUT
        gr.gemm_relu_debug_set(0, 0)
        c = gr.gemm_relu_streamk(a, b, workspace=ws)
        assert gr.status() == gr.OK
    finally:
        gr.gemm_relu_debug_force_kernel(0)
    rows = list(range(0, M, 97))
    want = np.concatenate([orc.gemm_relu_f16_rows(A, B, r, 1) for r in rows])
    assert_parity(host(c)[rows], want, abs_dot(A[rows], B), K, "streamk after timeout")


def test_pair_kernel_dropped_arrival_times_out_and_recovers(orc):
    M, N, K = 512, 1024, 512
    A, B = inputs.make(M, N, K, seed=10)
    a, b = dev(A), dev(B)
    gr.gemm_relu_debug_force_kernel(gr.FORCE_PAIR)
    try:
        gr.gemm_relu_debug_set(1, 20_000_000)
        gr.gemm_relu(a, b)
        assert gr.status() == gr.ERR_TIMEOUT
        gr.gemm_relu_debug_set(0, 0)
        c = gr.gemm_relu(a, b)
        assert gr.status() == gr.OK
        assert_parity(host(c), orc.gemm_relu_f16(A, B), abs_dot(A, B), K, "pair after timeout")
    finally:
        gr.gemm_relu_debug_force_kernel(0)
