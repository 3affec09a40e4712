"""GB300-native Ulysses sequence-parallel attention hot path.

The P sequence-parallel ranks are emulated inside one GPU: the all-to-all is a
relayout kernel, document boundaries are rebuilt from the gathered
position_ids, and varlen causal GQA attention (windows, per-head sinks) runs
forward and backward on the tcgen05 tensor core.  The product is the C library
``libusp.so`` (include/usp.h); ``binding`` exposes its calls to Python.
"""
from . import binding  # noqa: F401
from .binding import UspError, AttnParams  # noqa: F401

__all__ = ["binding", "UspError", "AttnParams"]
