"""GPU checks of lazy_copy_to_device, the SM-driven upload of a step's inputs from pinned host
memory: bit-exact copies at several sizes, and the source / destination kinds it refuses."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pk(lazylib, cuda_ok):
    import position_independent_kv_lazy_gb300 as m
    return m


@pytest.mark.parametrize("nbytes", [16, 4096 + 16, 921_600, 3 * 1024 * 1024 + 48, 64 << 20])
def test_copy_to_device_bit_exact(pk, nbytes):
    # sizes below one wave, a decode step's inputs, and large enough for the threads to loop
    rng = np.random.default_rng(nbytes)
    host = torch.from_numpy(rng.integers(0, 256, nbytes, dtype=np.uint8)).pin_memory()
    dev = torch.full((nbytes,), 7, dtype=torch.uint8, device="cuda")
    pk.lazy_copy_to_device(dev, host)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), host)


def test_copy_to_device_rejects(pk):
    dev = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    pinned = torch.zeros(4096, dtype=torch.uint8).pin_memory()
    pageable = torch.zeros(4096, dtype=torch.uint8)
    for dst, src in ((dev, pageable),              # pageable host source
                     (dev, dev.clone()),           # device source
                     (pinned.clone().pin_memory(), pinned),  # host destination
                     (dev[8:4088], pinned[8:4088])):         # 8-byte aligned only
        with pytest.raises(pk.LazyError) as e:
            pk.lazy_copy_to_device(dst, src)
        assert e.value.status == pk.LAZY_ERR_INVALID_ARG
    pk.lazy_copy_to_device(dev[:0], pinned[:0])  # nothing to copy
