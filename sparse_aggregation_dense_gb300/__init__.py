"""GB300-native partition-local GCN / GraphSAGE layer (forward and backward).

The product is the C-ABI library ``libgnn.so`` (declared in ``include/gnn.h``,
hand-written CUDA for sm_103a under ``csrc/``).  ``gnn`` is its thin ctypes
binding, ``partition_model`` drives one partition's epoch through it,
``multi_partition`` trains several partitions on one GPU, ``distributed``
one partition per process, and ``gat_model`` drives the graph-attention layers.
"""
from . import gnn  # noqa: F401
from .partition_model import PartitionModel, ld_for, padded  # noqa: F401
from .multi_partition import MultiPartitionTrainer  # noqa: F401
from .distributed import DistributedPartitionTrainer, ExchangePlan  # noqa: F401
from .gat_model import GatModel  # noqa: F401
