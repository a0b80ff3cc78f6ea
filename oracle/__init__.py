"""CPU oracle for the sorting path -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously-correct restatements of what the GPU library computes
(oracle.c, wrapped by ctypes in oracle.py).  Only tests/, the smoke check in
__graft_entry__ and bench.py's CPU-baseline leg may import this package; the
product package never does, and this package never imports the product.
"""
from .oracle import (  # noqa: F401
    SOURCE,
    Oracle,
    build,
    compile_source,
    default,
    f32_bits_to_ordered,
    ordered_to_f32_bits,
    f32_bits_to_ordered_array,
    ordered_to_f32_bits_array,
    num_passes,
    digit_histograms,
    exclusive_scan_bins,
    radix_sort_pairs,
    radix_sort_keys,
    compact_positive,
    segmented_sort,
    bitonic_network,
    radix2_three_pass,
)
