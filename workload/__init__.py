"""Seeded synthetic inputs for the decode-step KV path (shared by the CUDA path's
tests and bench and by the CPU oracle's callers). Holds no arithmetic of the
path itself."""
from .configs import (ADVERSARIAL, BY_NAME, D, D_LATENT, D_ROPE, DECODE_BATCH,
                      LARGE_BATCH, LONG_CONTEXT, ROW_BYTES, TINY, WORKLOADS,
                      Workload, get, scaled)
from .gen import (ScoreStream, bf16_to_f32, build_native, calibrate_rho,
                  ctx_lens, fill_host_kv, host_kv_rows, normal_bf16, queries)
