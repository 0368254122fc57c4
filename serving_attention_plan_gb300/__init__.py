"""GB300 (sm_103a) serving attention over a block-sparse-row paged KV-cache.

The compute path lives in a C-ABI shared library built from `csrc/`
(declared in `include/fi.h`); `binding` marshals arguments to it.  Importing
this package does not load the library: `binding.lib()` does, and fails loudly
when it is missing.
"""
