"""DsaInstall: the deferred pool refill and the group-end metadata update.

[GLM] §4.4: refill runs after the layer's selected rows are ready and off the
attention's critical path; the rows it installs are for later steps.
[GLM] §5 and §5.1: per layer, the missed entries are written into their
replacement slots of that layer's pool (FIFO eviction); the metadata update
(FIFO pointers, pool ids) happens once, at the group's last layer.

The rows installed are the host rows of the missed tokens; the selection
buffer holds the same bytes at the misses' first positions.
"""
import numpy as np


def dsa_install(pool_rows: np.ndarray, plan, host_rows: np.ndarray) -> None:
    """Write every installed miss's host row into its victim slot (in place)."""
    for t, v, keep in zip(plan.miss_ids, plan.victim, plan.install):
        if keep:
            pool_rows[int(v)] = host_rows[int(t)]


def metadata_update(tags: np.ndarray, fifo_ptr: np.ndarray, plan) -> None:
    """Tag every installed victim slot with its token; advance the pointers."""
    for t, v, keep in zip(plan.miss_ids, plan.victim, plan.install):
        if keep:
            tags[int(v)] = int(t)
    fifo_ptr[:] = plan.ptr_next
