"""GB300-native BEV pooling (depth-weighted scatter-reduce).

The compute path is the C-ABI library ``libbevpool.so`` (hand-written CUDA
for sm_103a, declared in ``include/bevpool.h``).  ``bevpool`` is its thin
ctypes binding; ``workloads`` draws seeded synthetic inputs.  Importing this
package loads nothing; importing ``bevpool`` loads the library and raises if
it has not been built.
"""
__all__ = ["bevpool", "workloads"]
