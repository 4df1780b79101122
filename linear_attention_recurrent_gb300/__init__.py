"""Recurrent linear-attention decode over a paged fp32 state pool, on GB300.

GDN (gated delta rule, scalar decay), KDA (per-key-channel decay) and
Lightning Attention: hand-written sm_103a kernels behind the C ABI in
include/lar.h (liblar.so, built in-tree by ``_build.build()``).  This package
is the thin torch-facing binding; see ``binding`` for the calls.
"""
from .binding import (LAR_BETA_RAW, LAR_DEVERR_ACCEPTED, LAR_DEVERR_READ_SLOT, LAR_DEVERR_SEQLEN,
                      LAR_DEVERR_TIMEOUT, LAR_DEVERR_WRITE_SLOT, LAR_GATE_RAW, LAR_QK_L2NORM, LAR_STATE_KV, LarError,
                      PreparedCall, StepGraph,
                      gdn_decode, gdn_decode_tokens, gdn_decode_varlen, kda_decode, kda_decode_tokens,
                      kda_decode_varlen, la_decode, la_decode_varlen, gdn_prefill, kda_prefill, la_prefill,
                      library_path, load)

__all__ = ["gdn_decode", "kda_decode", "la_decode", "gdn_decode_tokens", "kda_decode_tokens",
           "gdn_decode_varlen", "kda_decode_varlen", "la_decode_varlen", "gdn_prefill", "kda_prefill", "la_prefill",
           "PreparedCall", "StepGraph", "LarError", "load", "library_path", "LAR_QK_L2NORM", "LAR_GATE_RAW",
           "LAR_BETA_RAW", "LAR_STATE_KV", "LAR_DEVERR_READ_SLOT", "LAR_DEVERR_WRITE_SLOT", "LAR_DEVERR_ACCEPTED",
           "LAR_DEVERR_SEQLEN", "LAR_DEVERR_TIMEOUT"]
