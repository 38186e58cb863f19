"""Host-resident data on the GPU path (page "推测式 KV 编码无损压缩 KV 缓存最高可达约
4 倍", section "该方法的用途": compressed caches offloaded to host memory).

With unified addressing, pinned host memory is mapped into the device's
address space, so the kernels read their inputs and write their outputs in
host memory directly over the CPU-GPU link.  Encoding from and to host memory,
and decoding a host-resident container into host memory, must give the same
bytes as the device-resident path.
"""
import pytest
import torch

import synth
from gpu_helpers import device_views, gpu_codec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("name", ["qwen3-0.6b-bf16", "qwen3-8b-e4m3"])
def test_host_resident_inputs_container_and_output(name):
    spec = synth.WORKLOADS[name].scaled(name="host-" + name, L=2, H=2, T=600, calib_draws=2)
    w = synth.make(spec)
    codec = gpu_codec(w)
    kv_d, mu_d = device_views(w)
    ref, nref = codec.encode(kv_d, mu_d)
    ref = ref[:nref].cpu()

    kv_h = kv_d.cpu().pin_memory()
    mu_h = mu_d.cpu().pin_memory()
    box_h = torch.zeros(codec.max_bytes, dtype=torch.uint8).pin_memory()
    _, nb = codec.encode(kv_h, mu_h, out=box_h)          # kernels read and write host memory
    torch.cuda.synchronize()
    assert nb == nref and torch.equal(box_h[:nb], ref)

    out_h = torch.zeros_like(kv_h).pin_memory()
    codec.decode(box_h, nb, mu_h, out=out_h)             # host container -> host cache
    torch.cuda.synchronize()
    assert torch.equal(out_h, kv_h)

    out_d = codec.decode(box_h, nb, mu_d)                # host container -> device cache
    assert torch.equal(out_d, kv_d)
    t_h = codec.ideal_bits(kv_h, mu_h)
    t_d = codec.ideal_bits(kv_d, mu_d)
    assert t_h == t_d
