"""k6attn: joint-sequence attention for long-context video DiTs on GB300 (sm_103a).

The compute path is the C-ABI library `libk6attn.so` (CUDA kernels for
sm_103a); `video_dit_long_gb300.k6attn` is its thin ctypes binding.  Importing
this package loads nothing: the binding loads the library on first use and
raises if it is missing.
"""
