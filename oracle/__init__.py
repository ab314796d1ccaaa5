"""CPU oracle for the small-M routed-MoE layer (test infrastructure only).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The GPU library never imports it and shares no code
with it.  ``build()`` compiles ``moe_oracle.cpp`` into ``liboracle.so``;
``oracle.py`` holds the ctypes wrapper.
"""
