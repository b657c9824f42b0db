"""Routed MoE expert-parallel dispatch / combine for one GB300 GPU.

All W expert-parallel ranks live as blocks of one GPU's memory; the kernels
(sm_103a) sit behind the C-ABI in ``include/ep.h`` and this package binds it
for PyTorch tensors. See ``ep.EpContext``.
"""
from .ep import EpConfig, EpContext, DispatchOut, capacities, workspace_bytes  # noqa: F401
from ._lib import EpError  # noqa: F401
