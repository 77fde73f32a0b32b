"""fp64 CPU oracle for speculative-decoding verification.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference legs, never by the product library.
"""
from .spec_oracle import *  # noqa: F401,F403
from .spec_oracle import __all__ as _core_all
from .analysis import *  # noqa: F401,F403
from .analysis import __all__ as _analysis_all
from .rounds import *  # noqa: F401,F403
from .rounds import __all__ as _rounds_all
from .centroid import *  # noqa: F401,F403
from .centroid import __all__ as _centroid_all

__all__ = list(_core_all) + list(_analysis_all) + list(_rounds_all) + list(_centroid_all)
