"""The binding's marshalling checks: tensors the C ABI would read as plain pointers are
refused on the host when their device, dtype, layout or size cannot be right."""
import pytest
import torch

from deterministic_top_key_gb300 import binding


def _desc(T=6, Tkv=10, top_k=4):
    return binding.Desc(T, Tkv, [0, T], [0, Tkv], top_k)


def _bufs(T=6, Tkv=10, top_k=4, device="cpu"):
    q = torch.zeros((T, 64, 128), dtype=torch.bfloat16, device=device)
    k = torch.zeros((Tkv, 128), dtype=torch.bfloat16, device=device)
    w = torch.zeros((T, 64), dtype=torch.float32, device=device)
    ids = torch.zeros((T, top_k), dtype=torch.int32, device=device)
    sc = torch.zeros((T, top_k), dtype=torch.float32, device=device)
    return q, k, w, ids, sc


def _refused(desc, *bufs, match):
    with pytest.raises(binding.IndexerTopkError) as e:
        binding._check_buffers(desc, *bufs)
    assert e.value.status == binding.ITK_ERR_INVALID_ARGUMENT
    assert match in str(e.value)


def test_host_tensors_are_refused():
    _refused(_desc(), *_bufs(), match="not a CUDA device")


def test_eager_entry_refuses_before_calling_the_library():
    with pytest.raises(binding.IndexerTopkError) as e:
        binding.indexer_topk_eager(_desc(), *_bufs(), None)
    assert e.value.status == binding.ITK_ERR_INVALID_ARGUMENT


class _FakeCuda:
    """Stands in for a CUDA tensor on a host without a GPU (metadata only)."""

    def __init__(self, t, device="cuda:0", contiguous=True):
        self.t, self.device, self._c = t, torch.device(device), contiguous
        self.is_cuda, self.dtype = True, t.dtype

    def is_contiguous(self):
        return self._c

    def numel(self):
        return self.t.numel()


def _fake(bufs, device="cuda:0"):
    return [_FakeCuda(t, device=device) for t in bufs]


@pytest.fixture(autouse=True)
def current_device_is_cuda0(monkeypatch):
    """The library launches on the calling thread's current CUDA device; here that is a
    stand-in for cuda:0 (no GPU on this host)."""
    monkeypatch.setattr(binding, "_current_cuda_device", lambda: torch.device("cuda", 0))


def test_well_formed_buffers_pass():
    binding._check_buffers(_desc(), *_fake(_bufs()))
    q, k, w, ids, sc = _fake(_bufs())
    binding._check_buffers(_desc(), q, k, None, ids, sc)  # a missing buffer is the library's to report
    flat_k = _FakeCuda(torch.zeros(10 * 128 + 7, dtype=torch.bfloat16))
    binding._check_buffers(_desc(), q, flat_k, w, ids, sc)  # a flat buffer of enough elements


def test_wrong_dtype_layout_size_or_device_is_refused():
    q, k, w, ids, sc = _fake(_bufs())
    _refused(_desc(), _FakeCuda(torch.zeros((6, 64, 128), dtype=torch.float16)), k, w, ids, sc, match="dtype")
    _refused(_desc(), q, _FakeCuda(k.t, contiguous=False), w, ids, sc, match="not contiguous")
    _refused(_desc(), q, k, _FakeCuda(torch.zeros((5, 64))), ids, sc, match="want at least 384")
    _refused(_desc(), q, k, w, _FakeCuda(torch.zeros((6, 4), dtype=torch.int64)), sc, match="dtype")
    _refused(_desc(), q, k, w, ids, _FakeCuda(sc.t, device="cuda:1"), match="other buffers")
    _refused(_desc(top_k=8), q, k, w, ids, sc, match="want at least 48")


def test_buffers_on_another_device_than_the_current_one_are_refused():
    """Every buffer on cuda:1 while cuda:0 is current: the kernels would run on cuda:0 and
    reach the buffers as peer pointers, so the binding refuses before the C call."""
    _refused(_desc(), *_fake(_bufs(), device="cuda:1"), match="current CUDA device is cuda:0")
    binding._check_buffers(_desc(), *_fake(_bufs(), device="cuda:0"))
