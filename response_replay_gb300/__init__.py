"""GB300 response-replay hot path: paged prompt capture, replay attention forward and
backward over a read-only captured prompt, and the fused GRPO loss.

The computation lives in the CUDA library behind include/longstraw.h
(response_replay_gb300/_build/liblongstraw.so, built by ``build.py``).  ``binding``
is the ctypes binding with the C names; ``torch_api`` wraps it for torch tensors.
Importing this package does not load the library; the first call does, and fails
loudly if it has not been built.
"""
from . import binding  # noqa: F401
from .binding import (  # noqa: F401
    ls_capture_kv, ls_grpo_loss_fwd_bwd, ls_grpo_workspace, ls_last_device_error,
    ls_replay_attn_bwd, ls_replay_attn_bwd_workspace, ls_replay_attn_fwd,
    ls_replay_attn_fwd_workspace, ls_validate_page_table, ls_validate_page_table_workspace,
    LongstrawError,
)
