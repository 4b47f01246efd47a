"""LOCKS page-local key-summary sparse decode for GB300 (sm_103a).

The compute path is the CUDA library `liblocks.so` built from `csrc/`; the
Python side only marshals arguments (see `binding.py`).
"""
