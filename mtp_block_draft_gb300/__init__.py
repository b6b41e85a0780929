"""GB300-native (sm_103a) DMTP speculative-decoding round.

The round lives in the C-ABI library ``libdmtp.so`` (include/dmtp.h; the draft-depth
gate in include/dmtp_gate.h; the draft heads' token list in include/dmtp_vocab.h); this
package holds its CUDA sources (``csrc/``), the in-tree build (``build.py``) and the
ctypes binding (``binding.py``).
"""
from .binding import (DmtpError, DmtpGate, DmtpRound, DmtpVocabList, default_max_ctx,
                      load_library, make_config, make_weights)

__all__ = ["DmtpError", "DmtpGate", "DmtpRound", "DmtpVocabList", "default_max_ctx",
           "load_library", "make_config", "make_weights"]
