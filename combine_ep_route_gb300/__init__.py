"""Routed MoE expert-parallel dispatch / combine for one GB300 GPU.

All W expert-parallel ranks live as blocks of one GPU's memory; the kernels
(sm_103a) sit behind the C-ABI in ``include/ep.h`` and this package binds it
for PyTorch tensors. See ``ep.EpContext``.
"""
from .ep import (EpConfig, EpContext, DispatchOut, AgrsBuffers, agrs, alloc_agrs_buffers,  # noqa: F401
                 capacities, workspace_bytes)
from ._lib import EpError  # noqa: F401
