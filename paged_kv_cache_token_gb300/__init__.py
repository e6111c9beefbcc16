"""GB300-native paged-KV attention step (decode + chunked prefill) behind a C ABI.

The compute lives in ``libpkv.so`` (CUDA, sm_103a; declarations in include/pkv.h);
:mod:`.binding` marshals arguments to it.  :mod:`.scheduler` plans token-budget steps and
pages on the host; :mod:`.workloads` draws seeded synthetic inputs; :mod:`.runner` drives
steps on a device.  Submodules load lazily so host-only users need no GPU.
"""
__all__ = ["binding", "build", "runner", "scheduler", "workloads"]
__version__ = "0.1.0"
