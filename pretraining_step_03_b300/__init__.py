"""B300-native nanochat pretraining step: Python binding over ``libnc.so``."""
