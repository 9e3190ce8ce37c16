"""CPU oracle for the trellis-quantized projection (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package. The product library never imports, links or runs it.
"""
