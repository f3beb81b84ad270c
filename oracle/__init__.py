"""fp64 CPU oracle (test infrastructure only; see rlloss_oracle's header)."""
from .rlloss_oracle import *  # noqa: F401,F403
from .rlloss_oracle import (GMPO, GSPO_TOKEN, Problem, LossResult, row_stats, entropy_threshold,
                            gmpo_loss, gspo_token_loss, grads, loss_stage, fwd_bwd, as_f64,
                            as_i64, f32, logits_rows, entropy_direct, dlogits_rows, shard_state,
                            merge_states, shard_grads)
