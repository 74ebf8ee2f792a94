"""DsaServe: per layer, prepare the rows sparse attention reads.

[GLM] §5 and §5.1: every layer applies the group's shared plan to its own
full KV cache in host memory and to its own pool view on the device, and
produces the selection buffer that SFA consumes. Bytes are only copied: row j
of the selection is pool row src_map[j] for a hit and host row (-1 - src_map[j])
for a miss. A latent row here is 576 bf16 values (512 latent + 64 rope) kept
together, where the page keeps the two parts in separate tensors.
"""
import numpy as np


def dsa_serve(src_map, pool_rows: np.ndarray, host_rows: np.ndarray,
              ctx_len: int) -> np.ndarray:
    out = np.empty((len(src_map), pool_rows.shape[1]), dtype=pool_rows.dtype)
    for j, src in enumerate(src_map):
        src = int(src)
        if src >= 0:
            if src >= pool_rows.shape[0]:
                raise ValueError("pool slot out of range")
            out[j] = pool_rows[src]
        else:
            t = -1 - src
            if t >= ctx_len:
                raise ValueError("host row out of range")
            out[j] = host_rows[t]
    return out
