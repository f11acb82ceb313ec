"""Device-side failure reports on the GPU, made without faulting it.

genie-ai-runtime release v0.1.0-alpha.11 ("--int8-kv triage") traces a hang to a
path that fell back silently.  Here every wait of a decode block on its page
copies is bounded; when a wait gives up, the block skips the page, sets
INT8KV_DEVERR_TIMEOUT in the pool's device error word and the call completes.
The diagnostic kv_pool_test_expire_waits makes every such wait expire (the
stage barriers are armed for bytes that no copy brings, and no copy is issued,
so nothing is in flight when a block gives up); the test checks that the report
arrives, that the context stays usable, and that switching the diagnostic off
restores results equal to the oracle's.
"""

import pytest
import torch

from tests import gpu_util as gu
from tests.test_gpu_decode import _decode, _oracle, _setup

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.lib_ready()


def test_expired_copy_waits_are_reported_and_the_context_stays_usable():
    from int8_kv_cache_02_gb300 import binding
    lens = [700, 300]
    q, pt, dev, orc = _setup(70, 2, 16, 2, 256, 64, lens, 0, outliers=True)
    assert binding.kv_pool_read_device_error(dev) == 0
    binding.kv_pool_test_expire_waits(dev, 2000)
    for ns in (1, 4, 16):          # single pass, one cluster, the combine kernel
        _decode(dev, 0, q, lens, pt, n_splits=ns)
        err = binding.kv_pool_read_device_error(dev)
        assert err & binding.DEVERR_TIMEOUT, (ns, err)
    # the fused append waits on its page too: it gives up and skips the row
    k_new = torch.zeros((2, 2, 256), dtype=torch.float16, device="cuda")
    out = torch.empty((2, 16, 256), dtype=torch.float32, device="cuda")
    lens2 = torch.tensor([701, 301], dtype=torch.int32, device="cuda")
    binding.attn_decode_append_int8(dev, 0, q.cuda(), k_new, k_new, lens2, pt.cuda(), out,
                                    dev.decode_workspace(2, 16, 4), n_splits=4)
    assert binding.kv_pool_read_device_error(dev) & binding.DEVERR_TIMEOUT
    # off again: the same context gives the oracle's result and a clean error word
    binding.kv_pool_test_expire_waits(dev, 0)
    gu.assert_attention_close(_decode(dev, 0, q, lens, pt, n_splits=4), _oracle(orc, 0, q, lens, pt),
                              "after the expired waits")
    assert binding.kv_pool_read_device_error(dev) == 0


def test_expiry_needs_the_warp_level_kernel():
    from int8_kv_cache_02_gb300 import binding
    q, pt, dev, orc = _setup(71, 1, 8, 2, 64, 32, [100], 0, ps=16)   # CUDA-core kernel shape
    with pytest.raises(binding.Int8KVError) as e:
        binding.kv_pool_test_expire_waits(dev, 100)
    assert e.value.status == -6
