"""fp64 CPU oracle — test infrastructure only (tests, smoke check, benchmark CPU baseline).

The product path never imports this package.
"""
