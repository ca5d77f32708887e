"""Float64 CPU oracle for MLA decode -- test infrastructure only.

Importable by tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg.
The product library (head_latent_attention_29_b300) never imports it."""
from .mla_oracle import *  # noqa: F401,F403
