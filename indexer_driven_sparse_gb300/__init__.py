"""GB300 (sm_103a) indexer-driven sparse attention behind the libqsa.so C ABI.

Submodules: ``binding`` (ctypes marshalling of the qsa_* calls), ``pipeline``
(buffers and call sequences for a decode layer-step or a prefill chunk),
``inputs`` (seeded synthetic workloads), ``accounting`` (algorithmic bytes and
FLOPs), ``build`` (nvcc build of the library).
"""

__version__ = "0.1.0"
