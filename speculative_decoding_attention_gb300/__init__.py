"""Windowed-MTP decode attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libwm.so`` (CUDA, built from
``csrc/``); ``wm`` is its thin ctypes binding.  Importing this package loads
nothing; ``wm.load()`` (called by every binding function) loads the library and
fails loudly when it is missing.
"""
