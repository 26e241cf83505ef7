"""Owner-local Muon optimizer step (MatrixFSDP hot path) for one GB300 GPU.

``mfsdp``        the Python binding of the C ABI in ``include/mfsdp.h`` (libmfsdp.so);
``owner_step``   buffers + call sequence of one owner step on flat device buffers;
``build``        in-tree nvcc build of the library for sm_103a.
"""

__all__ = ["mfsdp", "owner_step", "build"]
