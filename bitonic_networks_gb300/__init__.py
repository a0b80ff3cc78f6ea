"""gsort: GB300-native stable LSD radix sort, stream compaction and segmented
bitonic sort, in hand-written CUDA for sm_103a behind a C ABI (libgsort.so).

The torch-facing wrappers live in `bitonic_networks_gb300.gsort`; they are
loaded on first attribute access so that importing the package (for example
to reach the input generators in `synth`) does not require the CUDA library.
"""
import importlib

__all__ = [
    "sort", "sort_keys", "sort_pairs", "compact_positive", "segmented_sort_", "segmented_sort",
    "partition", "split_sort",
    "digit_histograms", "GsortError", "library_path",
    "radix_workspace_bytes", "sort_workspace_bytes", "segmented_sort_workspace_bytes",
    "compact_workspace_bytes",
]


def __getattr__(name):
    if name in __all__:
        mod = importlib.import_module(".gsort", __name__)
        return getattr(mod, name)
    raise AttributeError(name)
