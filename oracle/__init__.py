"""CPU oracle (test infrastructure only): see ``oracle.kvq_oracle``.

Only the tests, the smoke check and the CPU-baseline leg of the benchmark may
import this package; the GPU library never does.
"""
from . import kvq_oracle  # noqa: F401
