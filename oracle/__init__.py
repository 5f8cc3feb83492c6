"""CPU oracle (fp64, numpy) for KV-cache importance scoring and pruning.

TEST INFRASTRUCTURE: importable only from the tests, the smoke check and the CPU
baseline leg of the benchmark.  The library's product path never imports it.
"""
from .kvs_oracle import *  # noqa: F401,F403
