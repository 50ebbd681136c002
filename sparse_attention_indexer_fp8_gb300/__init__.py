"""GB300-native FP8 lightning indexer: Python binding over the C-ABI library ``libidx.so``."""
