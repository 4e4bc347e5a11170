"""dsa_stage_copy on the GPU: byte-exact copies host(pinned) -> device, device ->
host(pinned) and device -> device at sizes with and without a ragged tail (not a
multiple of 16) up to the decode step's packed inputs; pageable host memory and
misaligned pointers are refused before launch. The step's outputs written straight
to page-locked host memory."""
import pytest
import torch

from dsa_sparse_attention_02_gb300 import _lib
from gpu_helpers import DEV

pytestmark = pytest.mark.gpu

SIZES = [1, 15, 16, 17, 4099, 1 << 16, 1770240 + 7]


@pytest.mark.parametrize("n", SIZES)
def test_stage_copy_is_byte_exact_every_direction(n):
    g = torch.Generator().manual_seed(n)
    src_h = torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g).pin_memory()
    dev = torch.full((n + 32,), 0xA5, dtype=torch.uint8, device=DEV)
    _lib.dsa_stage_copy(dev, src_h, n)
    torch.cuda.synchronize()
    assert torch.equal(dev[:n].cpu(), src_h)
    assert torch.all(dev[n:] == 0xA5)                      # nothing past the range
    back = torch.zeros(n, dtype=torch.uint8).pin_memory()
    _lib.dsa_stage_copy(back, dev, n)
    torch.cuda.synchronize()
    assert torch.equal(back, src_h)
    dev2 = torch.zeros(n, dtype=torch.uint8, device=DEV)
    _lib.dsa_stage_copy(dev2, dev, n)
    torch.cuda.synchronize()
    assert torch.equal(dev2.cpu(), src_h)


def test_stage_copy_refuses_pageable_and_misaligned():
    dev = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    pageable = torch.zeros(4096, dtype=torch.uint8)           # not page-locked
    with pytest.raises(_lib.DsaError) as e:
        _lib.dsa_stage_copy(dev, pageable, 4096)
    assert e.value.status == _lib.DSA_ERR_INVALID_ARG
    pinned = torch.zeros(4096, dtype=torch.uint8).pin_memory()
    with pytest.raises(_lib.DsaError) as e:
        _lib.dsa_stage_copy(dev[8:], pinned, 1024)          # 8-byte offset
    assert e.value.status == _lib.DSA_ERR_INVALID_ARG
    _lib.dsa_stage_copy(dev, pinned, 0)                      # zero bytes: no-op


@pytest.mark.parametrize("name", ["decode", "mtp"])
def test_step_writes_outputs_straight_to_page_locked_host_memory(name):
    """The step with O and LSE in page-locked host memory (written by the attention and
    combine kernels over the host link) gives the device step's outputs bit for bit;
    pageable host memory is refused before launch."""
    from dsa_sparse_attention_02_gb300 import inputs, runner
    wl = inputs.make_config(name, batch=8)
    dw = runner.DeviceWorkload(wl, DEV)
    dw.step()
    torch.cuda.synchronize()
    assert dw.check_error() == 0
    ref = dw.outputs.cpu()
    host_out = torch.full(dw.outputs.shape, 0x7F, dtype=dw.outputs.dtype).pin_memory()
    base, hbase = dw.outputs.data_ptr(), host_out.data_ptr()
    for a in dw.args:
        ha = _lib.dsa_step_args_t.from_buffer_copy(a)
        ha.out = hbase + (a.out - base)
        ha.lse = hbase + (a.lse - base)
        _lib.dsa_decode_step(ha, dw.ws)
    torch.cuda.synchronize()
    assert dw.check_error() == 0
    assert torch.equal(host_out, ref)
    pageable = torch.zeros(dw.outputs.shape, dtype=dw.outputs.dtype)
    ha = _lib.dsa_step_args_t.from_buffer_copy(dw.args[0])
    ha.out = pageable.data_ptr() + (dw.args[0].out - base)
    with pytest.raises(_lib.DsaError) as e:
        _lib.dsa_decode_step(ha, dw.ws)
    assert e.value.status == _lib.DSA_ERR_INVALID_ARG
