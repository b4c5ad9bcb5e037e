"""GB300-native tensor-parallel Transformer MLP block (forward and backward).

Importing the package loads nothing; ``binding`` opens the CUDA library on
first use and raises if it has not been built.
"""
