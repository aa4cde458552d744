"""The fp64 CPU oracle of the packed CTC loss (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library and never imports it.
"""

from .ctc_oracle import (build, ctc_loss_packed, ctc_loss_packed_logits, log_softmax_rows,  # noqa: F401
                         max_threads, oracle_batch, raw_nll_and_grad, reduce_losses, utterance_scales)
