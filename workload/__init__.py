"""Seeded synthetic inputs for paged decode: a counter-based value generator
(``workload.rng``) and the five workload definitions (``workload.configs``).

Shared by the GPU path, the tests and the oracle; holds no paged-attention
arithmetic (no block tables, slots, copies or softmax)."""
