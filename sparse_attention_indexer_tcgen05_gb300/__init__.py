"""GB300 (sm_103a) CSA Lightning-Indexer training step: score + top-k, full-CSA teacher, KL and the
sparse indexer backward, behind the C-ABI library ``libcsa_indexer.so``.

Importing the package loads nothing; ``from sparse_attention_indexer_tcgen05_gb300 import binding``
loads the CUDA library (and fails loudly if it has not been built).
"""
__all__ = ["binding", "synth"]
