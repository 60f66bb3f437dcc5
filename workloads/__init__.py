"""Seeded synthetic inputs for paged KV storage and paged attention.

Shared by the tests, the benchmark and the smoke check, on both sides of every parity
comparison.  It holds none of the method's arithmetic: no address rule, no slot mapping,
no store, no attention.  It draws numbers and hands out pages (a host page allocator in
the manner of TileInfer.jl's BlockManager), nothing else.
"""
from .gen import (BF16_NAN, Case, OutOfPages, PageAllocator, bf16_bits, build_case,
                  f32_from_bf16, normal_bf16)
from .configs import CONFIGS, config_case

__all__ = ["BF16_NAN", "Case", "OutOfPages", "PageAllocator", "bf16_bits", "build_case",
           "f32_from_bf16", "normal_bf16", "CONFIGS", "config_case"]
