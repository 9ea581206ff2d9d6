"""libmaskllm: MaskLLM's differentiable 2:4 mask layer on GB300 (sm_103a).

The compute lives in ``libmaskllm.so`` (hand-written CUDA behind a C ABI,
declared in ``include/maskllm.h``).  ``binding`` is the thin Python layer over
it; ``workloads`` draws the seeded synthetic inputs.
"""
__version__ = "0.1.0"
