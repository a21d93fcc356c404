"""CPU oracle (fp64) for predictor-gated activation-sparse FFN decode.

Test infrastructure only: the tests, the package smoke check and the
benchmark's CPU baseline call it; the product path never imports it.
"""
from .sffn_oracle import *  # noqa: F401,F403
from .sffn_oracle import OracleLayer, SparseResult  # noqa: F401
