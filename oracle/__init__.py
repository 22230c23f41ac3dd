"""CPU oracle of a batch-1 Llama decode step: TEST INFRASTRUCTURE ONLY.

Only tests/, the smoke check and the benchmark's CPU-baseline / reference
legs may import it; the CUDA package never does.  See oracle.h.
"""
