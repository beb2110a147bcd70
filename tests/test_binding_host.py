"""CPU-side checks of the Python binding's marshalling: buffers of one call must share
one CUDA device, and an explicit torch stream must belong to it.  The library launches
on the current device, so a pointer from another GPU would reach a kernel as a foreign
address; the binding refuses such a call on the host.  Only `.device` of each object is
read, so stand-ins with that attribute exercise the checks without a GPU."""
import types

import pytest


@pytest.fixture(scope="module")
def tdp():
    import __graft_entry__
    __graft_entry__.build()
    import blend_tdp_tile_gb300
    return blend_tdp_tile_gb300


def _on(dev):
    import torch
    return types.SimpleNamespace(device=torch.device(dev))


def test_buffers_on_one_device_pass(tdp):
    import torch
    named = [("X", _on("cuda:1")), ("P", None), ("Y", _on("cuda:1"))]
    assert tdp._common_device("tdp_split", named) == torch.device("cuda:1")


def test_no_buffers_gives_no_device(tdp):
    assert tdp._common_device("tdp_split", [("P", None)]) is None


def test_buffer_on_another_device_is_refused(tdp):
    named = [("X", _on("cuda:0")), ("Y", _on("cuda:1"))]
    with pytest.raises(ValueError, match="Y is on cuda:1 but X is on cuda:0"):
        tdp._common_device("tdp_split", named)


def test_stream_of_another_device_is_refused(tdp):
    import torch
    stream = types.SimpleNamespace(device=torch.device("cuda:1"), cuda_stream=1234)
    with pytest.raises(ValueError, match="stream is on cuda:1"):
        tdp._stream_handle("tdp_blend", stream, torch.device("cuda:0"))


def test_stream_of_the_same_device_passes(tdp):
    import torch
    stream = types.SimpleNamespace(device=torch.device("cuda:0"), cuda_stream=1234)
    assert tdp._stream_handle("tdp_blend", stream, torch.device("cuda:0")) == 1234
    assert tdp._stream_handle("tdp_blend", 99, torch.device("cuda:0")) == 99
