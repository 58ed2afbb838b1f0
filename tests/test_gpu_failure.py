"""Failure paths on the GPU without a fault: the library's bounded wait gives up, records
WQ_DEV_TIMEOUT and returns, and the context stays usable.

The probe (wq_test_wait_timeout) is one warp waiting on a shared-memory barrier that
nobody arrives on, with a 1 ms limit; it issues no copy and has no cluster peer, so
giving up leaves nothing in flight.  The same wait, with the arrival made first,
succeeds without the flag.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_linear_gb300 as wq
from weight_only_quantized_linear_gb300 import synth
from gpu_util import assert_within, bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    wq.build()


def test_bounded_wait_gives_up_and_reports_timeout(cuda_device):
    d = cuda_device
    st = torch.zeros(1, dtype=torch.int32, device=d)
    wq.wq_test_wait_timeout(1_000_000, arrive=False, dev_status=st)
    torch.cuda.synchronize()                       # the stream completes
    assert int(st.item()) == wq.WQ_DEV_TIMEOUT


def test_bounded_wait_completes_without_flag(cuda_device):
    d = cuda_device
    st = torch.zeros(1, dtype=torch.int32, device=d)
    wq.wq_test_wait_timeout(1_000_000, arrive=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_context_usable_after_timeout(cuda_device):
    """After a timeout the next linear call on the same stream gives correct results."""
    d = cuda_device
    st = torch.zeros(1, dtype=torch.int32, device=d)
    wq.wq_test_wait_timeout(1_000_000, arrive=False, dev_status=st)
    N, K, G = 512, 2048, 128
    rng = np.random.default_rng(3)
    packed = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scale = (rng.random((N, K // G)) * 0.018 + 0.002).astype(np.float32)
    zero = rng.integers(6, 10, (N, K // G), dtype=np.uint8)
    x = synth.normal_bf16((1, K), seed=4)
    st2 = torch.zeros(1, dtype=torch.int32, device=d)
    y = wq.wq_linear_int4_groups(x.to(d), torch.from_numpy(packed).to(d), torch.from_numpy(scale).to(d),
                                 torch.from_numpy(zero).to(d), None, G, dev_status=st2)
    torch.cuda.synchronize()
    assert int(st.item()) == wq.WQ_DEV_TIMEOUT and int(st2.item()) == 0
    yr, ad = oracle.linear_int4_groups(bf16_bits(x), packed, scale, zero, None, N, G)
    assert_within(y, yr, ad, "after timeout")


def test_wait_probe_rejects_long_limits(cuda_device):
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    with pytest.raises(wq.WQError) as e:
        wq.wq_test_wait_timeout(10 ** 9, arrive=False, dev_status=st)
    assert e.value.status == wq.WQ_EINVAL


@pytest.mark.parametrize("variant", [0, 1])
def test_stream_read_probe_runs(cuda_device, variant):
    """The read-only ceiling kernel reads the buffer and writes nothing."""
    d = cuda_device
    buf = torch.arange(3 * 1024 * 1024 // 4 + 4, dtype=torch.int32, device=d)
    sink = torch.zeros(1, dtype=torch.int32, device=d)
    for _ in range(3):
        wq.wq_bench_stream_read(buf, variant, sink)
    torch.cuda.synchronize()
    assert int(sink.item()) == 0
