"""CPU stand-ins for the CUDA calls bench.py makes, and a stub of liblowram.so that reports success.

Test infrastructure for the host-logic tests of bench.py (tests/test_bench_host.py) only.  install() runs in a
child process: tensors asked for on a CUDA device stay on the host, events and streams are inert, and every
library entry point returns LOWRAM_OK without touching memory (workspace queries answer 1 MiB).  What bench.py
prints under it is meaningless as a measurement.  The tests check only that every mode runs to the end through the
binding's argument checks and prints one JSON line with the keys its contract names.
"""
import contextlib
import types

import torch

_orig_to = torch.Tensor.to


def _is_cuda(a):
    return (isinstance(a, torch.device) and a.type == "cuda") or (isinstance(a, str) and a.startswith("cuda"))


def _to(self, *args, **kwargs):
    args = tuple(a for a in args if not _is_cuda(a))
    if _is_cuda(kwargs.get("device")):
        kwargs.pop("device")
    if not args and not kwargs:
        return self
    return _orig_to(self, *args, **kwargs)


def _host(fn):
    def w(*args, **kwargs):
        if _is_cuda(kwargs.get("device")):
            kwargs.pop("device")
        return fn(*args, **kwargs)
    return w


class _Event:
    def __init__(self, *a, **k):
        self.cuda_event = None

    def record(self, *a, **k):
        pass

    def synchronize(self):
        pass

    def elapsed_time(self, other):
        return 1.0


class _Stream:
    cuda_stream = 0

    def synchronize(self):
        pass

    def wait_stream(self, *a):
        pass

    def record_event(self, *a):
        return _Event()


class _Library:
    """Every entry point succeeds; size and flag outputs get plausible values."""

    def __getattr__(self, name):
        def fn(*args):
            if name.endswith("_workspace_size"):
                args[-1]._obj.value = 1 << 20
            elif name in ("lowram_decode_uses_tensor_cores", "lowram_get_error"):
                args[-1]._obj.value = 1 if name == "lowram_decode_uses_tensor_cores" else 0
            elif name == "lowram_last_error":
                return b""
            elif name == "lowram_version":
                return 10000
            return 0
        return fn


def install():
    for name in ("empty", "zeros", "ones", "full", "randn", "rand", "randint", "arange", "empty_like", "zeros_like",
                 "ones_like", "full_like", "tensor", "as_tensor", "randn_like", "linspace", "logspace", "eye",
                 "randperm"):
        setattr(torch, name, _host(getattr(torch, name)))
    gen = torch.Generator
    torch.Generator = lambda *a, **k: gen()
    torch.Tensor.to = _to
    torch.Tensor.cuda = lambda self, *a, **k: self
    torch.Tensor.pin_memory = lambda self, *a, **k: self
    torch.cuda.is_available = lambda: True
    torch.cuda.synchronize = lambda *a, **k: None
    torch.cuda.current_stream = lambda *a, **k: _Stream()
    torch.cuda.Event = _Event
    torch.cuda.set_device = lambda *a, **k: None
    torch.cuda._sleep = lambda *a, **k: None
    torch.cuda.empty_cache = lambda: None
    torch.cuda.device_count = lambda: 1
    torch.cuda.get_device_name = lambda *a, **k: "host stand-in"
    torch.cuda.get_device_properties = lambda *a, **k: types.SimpleNamespace(uuid="host", name="host stand-in",
                                                                             multi_processor_count=148)
    import decode_attention_19_b300.binding as B
    lib = _Library()
    B._load = lambda: lib
    B._lib = lib

    def _dev(*ts):
        for t in ts:
            if t is not None and not t.is_contiguous():
                raise ValueError("tensors must be contiguous")
    B._dev = _dev
    B._on = lambda dev: contextlib.nullcontext()
