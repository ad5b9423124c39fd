"""Test infrastructure: the fp64 CPU oracle of the Gemma 3 attention block.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The product path never does.
"""
