"""DSpark block-drafter proposal head + greedy verify for GB300 (sm_103a).

The computation runs in libdspark.so (hand-written CUDA behind the C ABI of
include/dspark.h).  This package is its thin Python binding:

  _abi      ctypes functions with the C entry points' names
  torch_io  marshalling of torch tensors (device memory, streams) into those calls
  build     in-tree nvcc build of the library

Importing the package does not load the library; the first call does, and fails
loudly if the library has not been built.
"""
from ._abi import (DSPARK_BF16, DSPARK_F32, DSPARK_OK, DSparkError, check,  # noqa: F401
                   dspark_config, dspark_device_status, dspark_head, dspark_last_error,
                   dspark_num_slots, dspark_outputs, dspark_propose,
                   dspark_propose_workspace_size, dspark_status_string, dspark_tree_verify,
                   dspark_verify, dspark_wait_selftest, lib)
