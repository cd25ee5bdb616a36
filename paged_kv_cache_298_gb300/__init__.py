"""Paged GQA decode attention for GB300 (sm_103a): a C-ABI CUDA library and its thin
Python binding.  The binding is loaded on first use (see ``binding``)."""
