"""Test helper: build (if needed) and import the library binding."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def binding():
    from int4_routed_expert_moe_gb300 import build
    build.build()
    from int4_routed_expert_moe_gb300 import moe
    return moe
