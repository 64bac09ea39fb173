"""CPU float64 oracle for CoSA sparse prefill (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import this
package.  It shares no code with the CUDA path.
"""
from .cosa_oracle import *  # noqa: F401,F403
from .cosa_oracle import (COMPUTED, SKIPPED, IGNORED, Params, decode_bf16, token_set, direct_output,
                          kap_request_head, kap_mask, osk_qblock, osk_all,
                          stage1_count, flag_grouped_order, request_keys, request_queries,
                          kap_pbar_rows, kap_sampled)
