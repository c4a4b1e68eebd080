"""The oracle: a plain, slow CPU reference of the MoE layer forward pass.

Test infrastructure only (tests, the smoke check and the benchmark's CPU
baseline); the product path never imports it."""
from .moe_ref import *  # noqa: F401,F403
