"""CPU float64 oracle for QSA gather-GQA sparse attention.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's
CPU-baseline leg use it to check and time the CUDA path.  The product library
never imports it, and it imports nothing from the product package.
"""
from .oracle import (ORACLE_DTYPES, OracleError, build, compress_keys, decode, latent_attention,  # noqa: F401
                     load, msa_attention, sparse_attention)
