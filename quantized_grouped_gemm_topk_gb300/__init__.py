"""GB300 (sm_103a) routed Mixture-of-Experts layer: top-k routing, on-device
dispatch, FP8 x NVFP4/MXFP8/MXFP4 grouped GEMMs with a fused SwiGLU + requantise
epilogue, combine, and the training backward. The compute lives in the CUDA
library ``libmoe.so`` (C ABI: include/moe.h); ``binding`` marshals torch
tensors into it."""
from . import binding  # noqa: F401
from .binding import *  # noqa: F401,F403
