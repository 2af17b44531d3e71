"""P-EAGLE parallel drafting step on GB300 (sm_103a): Python binding of libpeagle.so."""
from .binding import (Drafter, Expanded, PeError, pe_draft_forward, pe_expand_batch,  # noqa: F401
                      pe_get_device_error, pe_lmhead_argmax, pe_linear, pe_set_trace)
