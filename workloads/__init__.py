"""Seeded synthetic workloads for the MoE layer (sizes, seeds, input tensors)."""
from .configs import MoEConfig, TINY, OLMOE, SKEW, DSV3, DOMINO, ALL, BY_NAME  # noqa: F401
