"""Paged grouped-query attention decode step for GB300 (sm_103a).

The compute path is the C-ABI library libpdattn (include/pdattn.h, CUDA
sources in csrc/); ``binding`` marshals torch tensors into it.  Importing
``binding`` fails if the library has not been built.
"""
