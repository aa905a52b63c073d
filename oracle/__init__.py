"""CPU oracle (test infrastructure only; see prefill_oracle.py)."""
from .prefill_oracle import *  # noqa: F401,F403
from .prefill_oracle import OracleModel, decode_prompt, rel_l2  # noqa: F401
