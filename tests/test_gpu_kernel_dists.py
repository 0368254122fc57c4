"""GPU parity on the kernel-level length distributions: batch 16 with constant(1024), uniform(512-1024)
and Zipf lengths, decode and causal prefill.  Source: page "FlashInfer：面向 LLM 推理服务的高效可定制
注意力引擎", 实验与指标 (paper §4.2, kernel-level benchmarks)."""
import pytest

from oracle import attention as A
from serving_attention_plan_gb300 import workloads as W

from .gpu_helpers import assert_close, run_library, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from serving_attention_plan_gb300 import build
    build.build()
    assert torch_mod().cuda.is_available()


@pytest.mark.parametrize("name", [n for n in W.KERNEL_DIST_WORKLOADS if n.endswith("_decode")])
def test_decode_distributions(name):
    b = W.by_name(name)
    o, lse, ws = run_library(b)
    assert ws.info()[1] == 0
    ro, rl = A.batch_attention(b)
    assert_close(o, lse, ro, rl)


@pytest.mark.parametrize("name", [n for n in W.KERNEL_DIST_WORKLOADS if n.endswith("_prefill")])
def test_prefill_distributions_full(name):
    b = W.by_name(name)
    o, lse, ws = run_library(b)
    assert ws.info()[1] == 1
    ro, rl = A.batch_attention(b)
    assert_close(o, lse, ro, rl)
