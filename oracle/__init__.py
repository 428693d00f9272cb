"""CPU oracle (test infrastructure): fp64 restatement of the GPT forward pass.

Imported only by tests, the smoke check and the benchmark's CPU baseline.
"""
