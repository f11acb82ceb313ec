"""The Python binding fails loudly instead of falling back (CPU only).

The binding only marshals tensors into the C ABI: a missing library raises, and
a tensor that is not a contiguous CUDA tensor of the declared dtype is refused
before any call reaches the library.
"""

import pytest
import torch

from int8_kv_cache_02_gb300 import binding


class _Pool:
    """Stand-in for a KVPool: the checks below fire before its handle is used."""
    handle = None
    n_kv_heads, head_dim = 2, 64


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        binding.lib()


@pytest.mark.parametrize("t,err", [
    (torch.zeros(4, dtype=torch.float16), ValueError),            # on the host
    ([0.0] * 4, TypeError),                                        # not a tensor
])
def test_tensors_must_be_cuda_tensors(t, err):
    with pytest.raises(err):
        binding._dev(t, torch.float16, "q")


def test_calls_refuse_host_tensors_before_the_library():
    binding.lib()   # built in-tree; the refusals below happen in the marshalling
    q = torch.zeros((1, 2, 8, 64), dtype=torch.float16)
    lens = torch.zeros(1, dtype=torch.int32)
    pt = torch.zeros((1, 4), dtype=torch.int32)
    out = torch.zeros((1, 2, 8, 64), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA"):
        binding.attn_decode_multi_int8(_Pool(), 0, q, lens, pt, out, n_splits=1)
    with pytest.raises(ValueError, match="CUDA"):
        binding.attn_decode_int8(_Pool(), 0, q[:, 0], lens, pt, out[:, 0], n_splits=1)
