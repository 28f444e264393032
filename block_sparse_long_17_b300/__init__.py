"""QSA (Qwen Sparse Attention) for B300: a C-ABI CUDA library plus a thin binding.

``qsa`` holds the binding; ``workloads`` draws the seeded synthetic inputs;
``build`` compiles ``libqsa.so`` in place.
"""
