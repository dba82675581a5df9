"""CPU oracle for TIDE's layout-aware reduce-scatter and all-gather.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it.  The CUDA library never calls
it, and it shares no code with the library: the only module both sides use is
``synth`` (seeded input generation, no method arithmetic).
"""

from .tide_oracle import *  # noqa: F401,F403
