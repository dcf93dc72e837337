"""GB300 (sm_103a) hot path of VeriCache's lossless draft -> verify -> accept loop.

VeriCache: Turning Lossy KV Cache into Lossless LLM Inference
(gist.science/paper/2605.17613).  The compute lives in five CUDA shared
libraries behind the C ABI of ``include/vc.h``; ``_lib`` binds them with
ctypes (argument marshalling only) and ``runtime`` holds the device-side
state of a batch (draft cache, pinned full-KV store) and the round driver.

Importing ``_lib`` raises ImportError when the libraries have not been built:
there is no CPU fallback.
"""

__all__ = ["_lib", "runtime", "build"]
