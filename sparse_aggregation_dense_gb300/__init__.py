"""GB300-native partition-local GCN / GraphSAGE layer (forward and backward).

The product is the C-ABI library ``libgnn.so`` (declared in ``include/gnn.h``,
hand-written CUDA for sm_103a under ``csrc/``).  ``gnn`` is its thin ctypes
binding and ``partition_model`` drives one partition's epoch through it.
"""
from . import gnn  # noqa: F401
from .partition_model import PartitionModel, ld_for, padded  # noqa: F401
from .multi_partition import MultiPartitionTrainer  # noqa: F401
