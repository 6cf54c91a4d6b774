"""Staging a decode step's activations from page-locked host memory
(ovl_stage_activations) and writing outputs straight to page-locked host
memory: byte-exact copies at odd sizes and offsets, pageable memory refused
before anything is launched, and a chain of steps that stage into one device
buffer while earlier forwards still read it."""
import numpy as np
import pytest

import synth as S
from gpu_common import make_runtime, require_gpu, stage, torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes,offset", [(36864, 0), (16, 0), (15, 0), (1, 3), (1000003, 5), (70000, 16)])
def test_stage_copies_bytes_exactly(nbytes, offset):
    require_gpu()
    import quantized_base_lora_gb300 as q
    src = torch.from_numpy(np.random.default_rng(nbytes).integers(0, 256, nbytes + 32, dtype=np.uint8)).pin_memory()
    dst = torch.zeros(nbytes + 32, dtype=torch.uint8, device="cuda")
    st = q.ovl_stage_activations(dst.data_ptr() + offset, src.data_ptr() + offset, nbytes,
                                 int(torch.cuda.current_stream().cuda_stream))
    assert st == q.OVL_OK
    torch.cuda.synchronize()
    got = dst.cpu().numpy()
    want = src.numpy()
    assert np.array_equal(got[offset:offset + nbytes], want[offset:offset + nbytes])
    assert not got[:offset].any() and not got[offset + nbytes:].any()


def test_stage_refuses_pageable_memory_and_mismatched_alignment():
    require_gpu()
    import quantized_base_lora_gb300 as q
    pageable = np.zeros(4096, dtype=np.uint8)
    dst = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    pinned = torch.zeros(4096, dtype=torch.uint8).pin_memory()
    assert q.ovl_stage_activations(dst.data_ptr(), pageable.ctypes.data, 4096) == q.OVL_E_ARG
    assert q.ovl_stage_activations(dst.data_ptr() + 1, pinned.data_ptr(), 64) == q.OVL_E_ARG
    assert q.ovl_stage_activations(0, pinned.data_ptr(), 64) == q.OVL_E_ARG
    assert q.ovl_stage_activations(dst.data_ptr(), pinned.data_ptr(), 0) == q.OVL_OK
    torch.cuda.synchronize()


def test_chained_steps_stage_into_one_buffer_and_write_host_outputs():
    """Six steps, each staging its own x into the same device buffer and
    writing y into its own page-locked host buffer, issued back to back on one
    stream; every y equals the output of the same x run with device buffers."""
    require_gpu()
    import quantized_base_lora_gb300 as q
    rng = np.random.default_rng(7)
    m, n = 2048, 4096
    W = S.gaussian(rng, (m, n), 0.02)
    base = S.build_base(S.Q8_0, [(0, 0, W)])
    A = S.gaussian(rng, (16, n), 0.01)
    B = S.gaussian(rng, (m, 16), 0.01)
    rt = make_runtime(base, arena_bytes=64 << 20)
    h = stage(rt, S.build_adapter(base, [0], [16], [(A, B)]))
    assert rt.activate([h], [2.0])[0] == 0
    stream = torch.cuda.Stream()
    sh = int(stream.cuda_stream)
    xs = [S.to_bf16_bits(S.gaussian(rng, (1, n), 1.0)) for _ in range(6)]
    x_pin = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in xs]
    y_pin = [torch.full((1, m), float("nan")).pin_memory() for _ in xs]
    x_dev = torch.empty((1, n), dtype=torch.int16, device="cuda")
    for xp, yp in zip(x_pin, y_pin):
        assert q.ovl_stage_activations(x_dev.data_ptr(), xp.data_ptr(), x_dev.numel() * 2, sh) == 0
        assert q.ovl_linear_forward(rt.ctx, 0, x_dev.data_ptr(), q.OVL_BF16, 1, yp.data_ptr(), q.OVL_PATH_DUAL,
                                    0, 0, sh) == 0
    stream.synchronize()
    assert rt.check_device() == 0
    for x, yp in zip(xs, y_pin):
        xd = torch.from_numpy(x.view(np.int16)).cuda()
        yd = torch.empty((1, m), device="cuda")
        assert q.ovl_linear_forward(rt.ctx, 0, xd.data_ptr(), q.OVL_BF16, 1, yd.data_ptr(), q.OVL_PATH_DUAL,
                                    0, 0, int(torch.cuda.current_stream().cuda_stream)) == 0
        torch.cuda.synchronize()
        assert np.array_equal(yp.numpy().view(np.uint32), yd.cpu().numpy().view(np.uint32))
    rt.close()
