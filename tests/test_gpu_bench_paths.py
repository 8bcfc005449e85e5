"""The measurement paths of bench.py compute what they time: the streamed
end-to-end prefill (host inputs copied in, outputs copied out, three device
buffer sets on their own streams) hands back exactly the outputs of the same
prefill run on device-resident inputs."""
import pytest
import torch

import bench
import gated_deltanet_state_gb300 as gdn

pytestmark = pytest.mark.gpu


def test_streamed_end_to_end_outputs_equal_the_device_run():
    gdn.load_library()
    w = bench.PrefillWork(3, seq_len=512)          # 4 sequences x 512 tokens, 27B-shaped layer
    w.run()
    torch.cuda.synchronize()
    assert int(w.err.item()) == 0
    ref = w.o.cpu()
    w.o_host.zero_()
    ms = w.e2e_pipelined_ms(steps=4)
    assert ms > 0
    assert int(w.err.item()) == 0
    # the last step's outputs, copied to pinned host memory by the pipeline
    assert torch.equal(w.o_host, ref)
    assert w.h2d_bytes == sum(v.numel() * v.element_size() for v in w.host.values())
    assert w.d2h_bytes == ref.numel() * ref.element_size()
