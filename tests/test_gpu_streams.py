"""GPU: the library keeps no state between calls, so the same sequence of calls
issued on two streams at once (different inputs, outputs in separate buffers)
gives the same bits as each sequence run alone."""
import pytest
import torch

from test_gpu_graph import Step, _same

pytestmark = pytest.mark.gpu


def test_two_streams_at_once_match_one_at_a_time(ro):
    a, b = Step(ro, 0), Step(ro, 1)
    a.run()
    alone_a = a.snapshot()
    b.run()
    alone_b = b.snapshot()
    a.poison()
    b.poison()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        with torch.cuda.stream(s1):
            a.run()
        with torch.cuda.stream(s2):
            b.run()
    torch.cuda.synchronize()
    _same(alone_a, a.snapshot())
    _same(alone_b, b.snapshot())
    assert ro.library().rowops_pipeline_timeouts() == 0
