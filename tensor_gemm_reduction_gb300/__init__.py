"""GB300 (sm_103a) shard-reduction GEMM: AR, RS and AG modes behind a C ABI.

The compute path is the CUDA library built from ``csrc/``; ``binding`` wraps
its entry points with the same names. Importing this package does not load the
library; the first call does, and fails loudly if it has not been built.
"""
