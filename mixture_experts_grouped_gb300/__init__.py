"""GB300 (sm_103a) grouped mixture-of-experts expert-FFN path.

The compute lives in ``libmoe.so`` (CUDA kernels behind a C ABI, declared in
``include/moe.h``); :mod:`mixture_experts_grouped_gb300.moe` binds it with the
same function names. :mod:`mixture_experts_grouped_gb300.synth` draws the seeded
synthetic inputs. Importing the package loads nothing: the library is opened on
first use of the binding, and a missing library is an error, never a fallback.
"""
