"""Float64 CPU oracle for LongStraw branch replay.  TEST INFRASTRUCTURE ONLY.

Only tests/, the smoke check in __graft_entry__ and the CPU-baseline leg of bench.py may
import anything here.  The product path (the CUDA library and its Python binding) never
does, and shares no code with it.
"""
from .attention import (replay_response, replay_group, response_rows, merge_partials,  # noqa: F401
                        prompt_key_grads)
from .grpo import token_logp, grpo_loss, surrogate, finalize  # noqa: F401
