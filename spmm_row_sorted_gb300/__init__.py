"""GB300-native truly sparse linear layer (row-sorted COO SpMM, SDDMM, DST restructure).

Importing the package does not load the CUDA library; ``spmm_row_sorted_gb300.snack``
loads it on first use and fails loudly when it has not been built.
"""
